// Runtime side of the C ABI: plan creation (device query, schedule build and
// validation, upload of tables and RoPE angles, scratch allocation), decode
// launches of up to 64 steps, status readback and the measurement helpers.
// "Tiles: Scheduling LLM Decoding as a Graph of Tiles", "What the code
// contains": the runtime re-validates a plan, checks it was made for this
// worker binary and GPU, and runs up to 64 tokens per cooperative launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "tiles_internal.h"

namespace tiles {
cudaError_t megakernel_configure(int d, int G, int wbytes, int ak, int smem_bytes);
cudaError_t megakernel_occupancy(int d, int G, int wbytes, int ak, int smem_bytes, int *blocks_per_sm);
cudaError_t kv8_from_bf16_launch(const uint16_t *k, const uint16_t *v, int Z, int max_pos, int mp, int d,
                                 int n_pos, int8_t *kq, float *ks, float *mu, int8_t *vq, float *vs,
                                 cudaStream_t st);
cudaError_t quantize_rows_launch(const void *src, int rows, int cols, void *dst, float *scale,
                                 int row_step, int row0, int offset, cudaStream_t st);
cudaError_t megakernel_launch(const KernelParams &p, int n_ctas, int smem_bytes, cudaStream_t st);
cudaError_t copy_launch(void *dst, const void *src, size_t bytes, int n_ctas, cudaStream_t st);
cudaError_t barrier_launch(uint32_t *ctr, int rounds, unsigned long long *elapsed, uint32_t *status,
                           int n_ctas, cudaStream_t st);
}  // namespace tiles

using namespace tiles;

static_assert(sizeof(CUtensorMap) == sizeof(TensorMap) && alignof(CUtensorMap) <= alignof(TensorMap),
              "TensorMap must hold a CUtensorMap");

#include "plan_internal.h"

namespace {

template <typename T>
cudaError_t dalloc(tiles_plan_s *p, T **ptr, size_t bytes) {
    void *v = nullptr;
    cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
    if (e != cudaSuccess) return e;
    p->allocs.push_back(v);
    *ptr = reinterpret_cast<T *>(v);
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t v) { return (v + 255u) & ~(size_t)255u; }

// The block of device memory every launch starts by zeroing: argmax keys [64] |
// phase counters | x words [H] | a words [F] | o words [nq d] | Q/K/V words
// [rows] | split partial words [nq][S][2 + d].
struct SyncLayout {
    size_t ctr, xw, aw, ow, qkvw, partw, bytes;
};
SyncLayout sync_layout(const tiles_schedule_s &s) {
    const Geom &g = s.geom;
    SyncLayout l;
    l.ctr = (size_t)kMaxStepsPerLaunch * 8;
    l.xw = align256(l.ctr + (size_t)s.n_counters * kCounterStride * 4);
    l.aw = align256(l.xw + (size_t)g.H * 4);
    l.ow = align256(l.aw + (size_t)g.F * 4);
    l.qkvw = align256(l.ow + (size_t)g.qd * 4);
    l.partw = align256(l.qkvw + (size_t)g.qkv_rows * 8);
    l.bytes = align256(l.partw + (size_t)g.nq * g.kv_splits * (2 + g.d) * 8);
    return l;
}
size_t sync_block_bytes(const tiles_schedule_s &s) { return sync_layout(s).bytes; }
void place_sync_block(const tiles_schedule_s &s, uint8_t *base, KernelParams *p) {
    const SyncLayout l = sync_layout(s);
    p->keys = reinterpret_cast<unsigned long long *>(base);
    p->counters = reinterpret_cast<uint32_t *>(base + l.ctr);
    p->xw = reinterpret_cast<uint32_t *>(base + l.xw);
    p->aw = reinterpret_cast<uint32_t *>(base + l.aw);
    p->ow = reinterpret_cast<uint32_t *>(base + l.ow);
    p->qkvw = reinterpret_cast<unsigned long long *>(base + l.qkvw);
    p->partw = reinterpret_cast<unsigned long long *>(base + l.partw);
}

// RoPE inverse frequencies theta^(-2j/d) in FP64, with the published llama3
// rule when enabled: wavelength 2 pi / w below orig/high keeps w, above
// orig/low divides it by the factor, between the two blends linearly in
// orig/wavelength.
void rope_inv_freq(const tiles_model_desc &d, std::vector<double> &w) {
    const int h = d.head_dim / 2;
    w.resize(h);
    for (int j = 0; j < h; ++j) {
        double f = std::pow(d.rope_theta, -(2.0 * j) / d.head_dim);
        if (d.rope_scaling == 1) {
            const double wl = 2.0 * M_PI / f;
            const double lo_wl = d.rs_orig_max / d.rs_low, hi_wl = d.rs_orig_max / d.rs_high;
            if (wl > lo_wl) {
                f = f / d.rs_factor;
            } else if (wl >= hi_wl) {
                const double sm = (d.rs_orig_max / wl - d.rs_low) / (d.rs_high - d.rs_low);
                f = (1.0 - sm) * (f / d.rs_factor) + sm * f;
            }
        }
        w[j] = f;
    }
}

tiles_status_t cuda_fail(cudaError_t e) {
    (void)e;
    return TILES_ERR_CUDA;
}

}  // namespace

extern "C" {

tiles_status_t tiles_plan_create(const tiles_model_desc *desc, const tiles_weights *w,
                                 const tiles_plan_opts *opts, tiles_plan_t *out) {
    if (!desc || !w || !out || !w->embed || !w->final_norm || !w->layers) return TILES_ERR_INVALID_ARG;
    *out = nullptr;
    tiles_plan_opts o = opts ? *opts : default_opts();
    if (o.timeout_ms < 0) return TILES_ERR_INVALID_ARG;
    // weights: present, 16-byte aligned
    if (!aligned16(w->embed) || !aligned16(w->final_norm)) return TILES_ERR_INVALID_ARG;
    for (int l = 0; l < desc->n_layers; ++l) {
        const tiles_layer_weights &lw = w->layers[l];
        const void *req[] = {lw.attn_norm, lw.wq, lw.wk, lw.wv, lw.wo, lw.ffn_norm, lw.w_gate, lw.w_up, lw.w_down};
        for (const void *q : req)
            if (!q || !aligned16(q)) return TILES_ERR_INVALID_ARG;
        if (desc->qk_norm && (!lw.q_norm || !lw.k_norm)) return TILES_ERR_INVALID_ARG;
    }

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!prop.cooperativeLaunch) return TILES_ERR_UNSUPPORTED;
    int smem_limit = (int)prop.sharedMemPerBlockOptin;
    if (smem_limit > kSmemLimit) smem_limit = kSmemLimit;
    int n_ctas = o.n_ctas > 0 ? o.n_ctas : prop.multiProcessorCount;
    if (n_ctas > prop.multiProcessorCount) return TILES_ERR_INVALID_ARG;

    auto *plan = new tiles_plan_s();
    plan->device = dev;
    plan->sm_count = prop.multiProcessorCount;
    plan->cc_major = prop.major;
    plan->cc_minor = prop.minor;
    std::string why;
    tiles_status_t st = build_schedule(*desc, o, n_ctas, smem_limit, &plan->sched, &why);
    if (st == TILES_OK) st = validate_schedule(plan->sched, &why);
    if (st != TILES_OK) {
        delete plan;
        return st;
    }
    const Geom &g = plan->sched.geom;

    // the worker must fit one CTA per SM at this shared-memory size (co-residency)
    e = megakernel_configure(g.d, g.G, g.wbytes, attn_kind(g), g.smem_bytes);
    int occ = 0;
    if (e == cudaSuccess) e = megakernel_occupancy(g.d, g.G, g.wbytes, attn_kind(g), g.smem_bytes, &occ);
    if (e != cudaSuccess || occ < 1) {
        delete plan;
        return e != cudaSuccess ? TILES_ERR_CUDA : TILES_ERR_UNSUPPORTED;
    }

    KernelParams &p = plan->base;
    std::memset(&p, 0, sizeof(p));
    p.g = g;
    p.eps = desc->rms_eps;
    p.attn_scale = (float)(1.0 / std::sqrt((double)g.d));
    p.qk_norm = desc->qk_norm;
    p.final_ctr = plan->sched.final_ctr;
    p.final_mul = plan->sched.final_mul;
    p.embed = reinterpret_cast<const uint16_t *>(w->embed);
    p.final_norm = reinterpret_cast<const uint16_t *>(w->final_norm);
    p.timeout_ns = (unsigned long long)(o.timeout_ms > 0 ? o.timeout_ms : 2000) * 1000000ull;
    // L2 lookahead is off unless asked for: on GB300 it competes with the ring
    // copies for the TMA unit and measured slower at every distance tried
    p.l2_prefetch_bytes = o.l2_prefetch_kb > 0 ? (unsigned long long)o.l2_prefetch_kb * 1024ull : 0ull;
    p.l2_prefetch_ns_per_4k = o.l2_prefetch_gbs > 0 ? (4096ull + (unsigned)o.l2_prefetch_gbs - 1) / (unsigned)o.l2_prefetch_gbs : 0ull;
    p.ring_off = kCtlBytes;
    p.vec_off = kCtlBytes + g.ring_slots * g.slot_bytes;
    p.res_off = g.res_off;
    auto fail = [&](cudaError_t ce) {
        tiles_plan_destroy(plan);
        return cuda_fail(ce);
    };
    tiles_task *d_tasks;
    int32_t *d_off;
    LayerPtrs *d_layers;
    if ((e = dalloc(plan, &d_tasks, plan->sched.tasks.size() * sizeof(tiles_task))) != cudaSuccess) return fail(e);
    if ((e = dalloc(plan, &d_off, plan->sched.offsets.size() * sizeof(int32_t))) != cudaSuccess) return fail(e);
    if ((e = dalloc(plan, &d_layers, (size_t)g.L * sizeof(LayerPtrs))) != cudaSuccess) return fail(e);
    std::vector<LayerPtrs> lp(g.L);
    const size_t H2 = (size_t)g.H * 2;
    for (int l = 0; l < g.L; ++l) {
        const tiles_layer_weights &lw = w->layers[l];
        LayerPtrs &L = lp[l];
        L.attn_norm = (const uint16_t *)lw.attn_norm;
        L.q_norm = (const uint16_t *)lw.q_norm;
        L.k_norm = (const uint16_t *)lw.k_norm;
        L.ffn_norm = (const uint16_t *)lw.ffn_norm;
        L.s_qkv = L.s_o = L.s_gu = L.s_down = nullptr;
        if (g.wbytes == 2) {
            // packed BF16 copies ("TilePlan ... packs the weights"): [Wq; Wk; Wv]
            // contiguous, and Wg / Wu interleaved by row, so each ring chunk is one bulk copy
            uint8_t *qkv, *gu;
            if ((e = dalloc(plan, &qkv, (size_t)g.qkv_rows * H2)) != cudaSuccess) return fail(e);
            if ((e = dalloc(plan, &gu, (size_t)g.F * 2 * H2)) != cudaSuccess) return fail(e);
            if ((e = cudaMemcpy(qkv, lw.wq, (size_t)g.qd * H2, cudaMemcpyDeviceToDevice)) != cudaSuccess ||
                (e = cudaMemcpy(qkv + (size_t)g.qd * H2, lw.wk, (size_t)g.kvd * H2, cudaMemcpyDeviceToDevice)) != cudaSuccess ||
                (e = cudaMemcpy(qkv + (size_t)(g.qd + g.kvd) * H2, lw.wv, (size_t)g.kvd * H2, cudaMemcpyDeviceToDevice)) !=
                    cudaSuccess ||
                (e = cudaMemcpy2D(gu, 2 * H2, lw.w_gate, H2, H2, g.F, cudaMemcpyDeviceToDevice)) != cudaSuccess ||
                (e = cudaMemcpy2D(gu + H2, 2 * H2, lw.w_up, H2, H2, g.F, cudaMemcpyDeviceToDevice)) != cudaSuccess)
                return fail(e);
            L.qkv = qkv;
            L.gu = gu;
            L.o = (const uint8_t *)lw.wo;
            L.down = (const uint8_t *)lw.w_down;
        } else {
            // INT8 codes and per-row scales, quantized straight into the packed layouts
            uint8_t *qkv, *o, *gu, *down;
            float *sqkv, *so, *sgu, *sdown;
            if ((e = dalloc(plan, &qkv, (size_t)g.qkv_rows * g.H)) != cudaSuccess ||
                (e = dalloc(plan, &o, (size_t)g.H * g.qd)) != cudaSuccess ||
                (e = dalloc(plan, &gu, (size_t)2 * g.F * g.H)) != cudaSuccess ||
                (e = dalloc(plan, &down, (size_t)g.H * g.F)) != cudaSuccess ||
                (e = dalloc(plan, &sqkv, (size_t)g.qkv_rows * 4)) != cudaSuccess ||
                (e = dalloc(plan, &so, (size_t)g.H * 4)) != cudaSuccess ||
                (e = dalloc(plan, &sgu, (size_t)2 * g.F * 4)) != cudaSuccess ||
                (e = dalloc(plan, &sdown, (size_t)g.H * 4)) != cudaSuccess)
                return fail(e);
            if ((e = quantize_rows_launch(lw.wq, g.qd, g.H, qkv, sqkv, 1, 0, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.wk, g.kvd, g.H, qkv, sqkv, 1, g.qd, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.wv, g.kvd, g.H, qkv, sqkv, 1, g.qd + g.kvd, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.wo, g.H, g.qd, o, so, 1, 0, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.w_gate, g.F, g.H, gu, sgu, 2, 0, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.w_up, g.F, g.H, gu, sgu, 2, 1, kCodeOffset, 0)) != cudaSuccess ||
                (e = quantize_rows_launch(lw.w_down, g.H, g.F, down, sdown, 1, 0, kCodeOffset, 0)) != cudaSuccess)
                return fail(e);
            L.qkv = qkv;
            L.o = o;
            L.gu = gu;
            L.down = down;
            L.s_qkv = sqkv;
            L.s_o = so;
            L.s_gu = sgu;
            L.s_down = sdown;
        }
    }
    // the LM head streams the tied embedding, or its INT8 codes
    p.lm = (const uint8_t *)w->embed;
    p.lm_s = nullptr;
    if (g.wbytes == 1) {
        uint8_t *lm;
        float *lms;
        if ((e = dalloc(plan, &lm, (size_t)g.V * g.H)) != cudaSuccess ||
            (e = dalloc(plan, &lms, (size_t)g.V * 4)) != cudaSuccess ||
            (e = quantize_rows_launch(w->embed, g.V, g.H, lm, lms, 1, 0, kCodeOffset, 0)) != cudaSuccess ||
            (e = cudaDeviceSynchronize()) != cudaSuccess)
            return fail(e);
        p.lm = lm;
        p.lm_s = lms;
    }
    {
        // the validated table, or (test hook) with CTA 0's first wait on a target
        // no launch reaches (counters stay far below 2^30)
        std::vector<tiles_task> up = plan->sched.tasks;
        if ((o.flags & TILES_FLAG_INJECT_STALL) && !up.empty() && plan->sched.offsets[1] > 0 &&
            up[0].wait_ctr != TILES_NO_COUNTER)
            up[0].wait_add += 0x40000000u;
        e = cudaMemcpy(d_tasks, up.data(), up.size() * sizeof(tiles_task), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess)
        e = cudaMemcpy(d_off, plan->sched.offsets.data(), plan->sched.offsets.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_layers, lp.data(), (size_t)g.L * sizeof(LayerPtrs), cudaMemcpyHostToDevice);
    plan->layers_host = lp;
    if (e != cudaSuccess) return fail(e);
    p.tasks = d_tasks;
    p.offsets = d_off;
    p.layers = d_layers;

    // RoPE cos/sin [max_pos][d/2]: angle pos * w_j in FP64, rounded to FP32
    {
        std::vector<double> inv;
        rope_inv_freq(*desc, inv);
        const int h = g.d / 2;
        std::vector<float> c((size_t)g.max_pos * h), s((size_t)g.max_pos * h);
        for (int pos = 0; pos < g.max_pos; ++pos)
            for (int j = 0; j < h; ++j) {
                const double a = (double)pos * inv[j];
                c[(size_t)pos * h + j] = (float)std::cos(a);
                s[(size_t)pos * h + j] = (float)std::sin(a);
            }
        float *dc, *ds;
        if ((e = dalloc(plan, &dc, c.size() * 4)) != cudaSuccess) return fail(e);
        if ((e = dalloc(plan, &ds, s.size() * 4)) != cudaSuccess) return fail(e);
        if ((e = cudaMemcpy(dc, c.data(), c.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess) return fail(e);
        if ((e = cudaMemcpy(ds, s.data(), s.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess) return fail(e);
        p.rope_cos = dc;
        p.rope_sin = ds;
    }
    // scratch
    // one memset per launch clears: argmax keys | phase counters | tagged activations
    // (tag 0 is never written, so nothing of an earlier launch reads as ready)
    plan->sync_bytes = sync_block_bytes(plan->sched);
    uint8_t *sync;
    if ((e = dalloc(plan, &sync, plan->sync_bytes)) != cudaSuccess) return fail(e);
    plan->d_keys = reinterpret_cast<unsigned long long *>(sync);
    p.keys = plan->d_keys;
    place_sync_block(plan->sched, sync, &p);
    if ((e = dalloc(plan, &p.status, 16)) != cudaSuccess) return fail(e);
    if ((e = cudaMemset(p.status, 0, 16)) != cudaSuccess) return fail(e);
    if ((e = dalloc(plan, &plan->d_prompt_stage, (size_t)g.max_pos * 4)) != cudaSuccess) return fail(e);
    if ((e = dalloc(plan, &plan->d_tokens_stage, (size_t)g.max_pos * 4)) != cudaSuccess) return fail(e);
    *out = plan;
    return TILES_OK;
}

void tiles_plan_destroy(tiles_plan_t plan) {
    if (!plan) return;
    for (void *v : plan->allocs) cudaFree(v);
    for (void *v : plan->fwd.allocs) cudaFree(v);
    delete plan;
}

tiles_status_t tiles_plan_set_trace(tiles_plan_t plan, void *trace, int32_t steps) {
    if (!plan || steps < 0 || (steps > 0 && !trace)) return TILES_ERR_INVALID_ARG;
    int mt = 0;
    for (int c = 0; c < plan->sched.n_ctas; ++c)
        mt = std::max(mt, plan->sched.offsets[c + 1] - plan->sched.offsets[c]);
    plan->base.trace = steps > 0 ? reinterpret_cast<unsigned long long *>(trace) : nullptr;
    plan->base.trace_steps = steps;
    plan->base.trace_tasks = mt;
    return TILES_OK;
}

tiles_status_t tiles_plan_get_info(tiles_plan_t plan, tiles_plan_info *info) {
    if (!plan) return TILES_ERR_INVALID_ARG;
    return tiles_schedule_get_info(&plan->sched, info);
}

tiles_status_t plan_check_device(tiles_plan_t plan) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TILES_ERR_CUDA;
    if (dev != plan->device) return TILES_ERR_DEVICE_MISMATCH;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TILES_ERR_CUDA;
    if (sms != plan->sm_count) return TILES_ERR_DEVICE_MISMATCH;
    return TILES_OK;
}

// cuTensorMapEncodeTiled, through the runtime's driver entry point (the
// library links only the static CUDA runtime)
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}


// TMA descriptors of this call's K and V caches: [L n_kv][max_pos][d] BF16,
// boxes of kv_block positions x 64 dims (a 128-dim head takes two boxes per
// chunk), 128-byte swizzle so the tensor-core fragment loads of the attention
// tiles are free of bank conflicts; positions past max_pos read as zero.
static tiles_status_t encode_kv_maps(const Geom &g, void *k_cache, void *v_cache, KernelParams *p) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return TILES_ERR_CUDA;
    const cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.max_pos, (cuuint64_t)g.L * (cuuint64_t)g.nkv};
    const cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.max_pos * (cuuint64_t)g.d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)g.kv_block, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    void *ptrs[2] = {k_cache, v_cache};
    for (int i = 0; i < 2; ++i) {
        CUtensorMap m;
        if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptrs[i], dims, strides, box, elem_strides,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TILES_ERR_CUDA;
        std::memcpy(&p->kv_map[i], &m, sizeof m);
    }
    return TILES_OK;
}

// The INT8 cache's two buffers (layout stated with tiles_kv8_layout).
static void kv8_layout_of(int Z, int max_pos, int d, tiles_kv8_layout *o) {
    auto up = [](int64_t v) { return (v + 255) / 256 * 256; };
    const int64_t mp = ((int64_t)max_pos + 15) / 16 * 16;
    o->pos_stride = (int32_t)mp;
    o->k_scale_off = up((int64_t)Z * mp * d);
    o->k_mu_off = up(o->k_scale_off + (int64_t)Z * mp * 4);
    o->k_bytes = o->k_mu_off + (int64_t)Z * d * 4;
    o->v_scale_off = up((int64_t)Z * d * mp);
    o->v_bytes = o->v_scale_off + (int64_t)Z * mp * 4;
}

// TMA descriptors of an INT8 cache: key codes [Z][MP][d] (box kv_block x d),
// value codes [Z][d][MP] (box d x kv_block), each swizzled by its row length
// (64 or 128 bytes) so the fragment loads spread over the banks, and the
// scales [Z][MP] (box kv_block). Positions past MP read as zero.
static tiles_status_t encode_kv8_maps(const Geom &g, void *k8, void *v8, KernelParams *p) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return TILES_ERR_CUDA;
    tiles_kv8_layout lay;
    kv8_layout_of(g.L * g.nkv, g.max_pos, g.d, &lay);
    const cuuint64_t Z = (cuuint64_t)g.L * (cuuint64_t)g.nkv, mp = (cuuint64_t)lay.pos_stride, d = (cuuint64_t)g.d;
    const cuuint32_t kvb = (cuuint32_t)g.kv_block, ones[3] = {1, 1, 1};
    auto sw = [](cuuint64_t row_bytes) {
        return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    };
    CUtensorMap m[4];
    {
        const cuuint64_t dims[3] = {d, mp, Z}, strides[2] = {d, mp * d};
        const cuuint32_t box[3] = {(cuuint32_t)d, kvb, 1};
        if (enc(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, k8, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                sw(d), CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TILES_ERR_CUDA;
    }
    {
        const cuuint64_t dims[3] = {mp, d, Z}, strides[2] = {mp, d * mp};
        const cuuint32_t box[3] = {kvb, (cuuint32_t)d, 1};
        if (enc(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, v8, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                sw(kvb), CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TILES_ERR_CUDA;
    }
    void *scales[2] = {static_cast<char *>(k8) + lay.k_scale_off, static_cast<char *>(v8) + lay.v_scale_off};
    for (int i = 0; i < 2; ++i) {
        const cuuint64_t dims[2] = {mp, Z}, strides[1] = {mp * 4};
        const cuuint32_t box[2] = {kvb, 1};
        if (enc(&m[2 + i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, scales[i], dims, strides, box, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TILES_ERR_CUDA;
    }
    std::memcpy(p->kv_map, m, sizeof m);
    p->k_cache = p->v_cache = nullptr;
    p->kq8 = static_cast<int8_t *>(k8);
    p->ks8 = reinterpret_cast<float *>(static_cast<char *>(k8) + lay.k_scale_off);
    p->mu8 = reinterpret_cast<const float *>(static_cast<char *>(k8) + lay.k_mu_off);
    p->vq8 = static_cast<int8_t *>(v8);
    p->vs8 = reinterpret_cast<float *>(static_cast<char *>(v8) + lay.v_scale_off);
    return TILES_OK;
}

// The caches of one decode call: pointers and TMA descriptors in p.
static tiles_status_t bind_caches(const Geom &g, void *k_cache, void *v_cache, KernelParams *p) {
    if (g.kv8) return encode_kv8_maps(g, k_cache, v_cache, p);
    p->k_cache = reinterpret_cast<uint16_t *>(k_cache);
    p->v_cache = reinterpret_cast<uint16_t *>(v_cache);
    return encode_kv_maps(g, k_cache, v_cache, p);
}

tiles_status_t tiles_decode(tiles_plan_t plan, void *k_cache, void *v_cache, const int32_t *prompt,
                            int32_t n_prompt, int32_t start_pos, int32_t n_new, void *stream,
                            int32_t *out_tokens, float *out_logits) {
    if (!plan || !k_cache || !v_cache || !prompt || n_prompt < 1 || n_new < 0 || start_pos < 0)
        return TILES_ERR_INVALID_ARG;
    if (n_new > 0 && !out_tokens) return TILES_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return TILES_ERR_INVALID_ARG;
    const Geom &g = plan->sched.geom;
    const long long steps = (long long)n_prompt - 1 + n_new;
    if (steps == 0) return TILES_OK;
    if ((long long)start_pos + steps > g.max_pos) return TILES_ERR_CAPACITY;
    tiles_status_t st = plan_check_device(plan);
    if (st != TILES_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    KernelParams p = plan->base;
    if ((st = bind_caches(g, k_cache, v_cache, &p)) != TILES_OK) return st;
    p.prompt = prompt;
    p.n_prompt = n_prompt;
    p.out_tokens = out_tokens;
    p.out_logits = out_logits;
    for (long long s0 = 0; s0 < steps; s0 += kMaxStepsPerLaunch) {
        const int n = (int)(steps - s0 < kMaxStepsPerLaunch ? steps - s0 : kMaxStepsPerLaunch);
        p.step0 = (int)s0;
        p.pos0 = start_pos + (int)s0;
        p.n_steps = n;
        cudaError_t e = cudaMemsetAsync(plan->d_keys, 0, plan->sync_bytes, cs);
        if (e == cudaSuccess) e = megakernel_launch(p, plan->sched.n_ctas, g.smem_bytes, cs);
        if (e != cudaSuccess) return TILES_ERR_CUDA;
    }
    return TILES_OK;
}

tiles_status_t tiles_status(tiles_plan_t plan, void *stream) {
    if (!plan) return TILES_ERR_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return TILES_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, plan->base.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return TILES_ERR_CUDA;
    if (word) {
        if (cudaMemset(plan->base.status, 0, 4) != cudaSuccess) return TILES_ERR_CUDA;
    }
    if (word & kDevBounds) return TILES_ERR_DEVICE_BOUNDS;
    if (word & kDevTimeout) return TILES_ERR_TIMEOUT;
    return TILES_OK;
}

tiles_status_t tiles_decode_host(tiles_plan_t plan, void *k_cache, void *v_cache,
                                 const int32_t *prompt_host, int32_t n_prompt, int32_t start_pos,
                                 int32_t n_new, void *stream, int32_t *out_tokens_host,
                                 float *out_logits_host) {
    if (!plan || !prompt_host || n_prompt < 1 || n_new < 0 || start_pos < 0) return TILES_ERR_INVALID_ARG;
    if (n_new > 0 && !out_tokens_host) return TILES_ERR_INVALID_ARG;
    const Geom &g = plan->sched.geom;
    const long long steps = (long long)n_prompt - 1 + n_new;
    if ((long long)start_pos + steps > g.max_pos) return TILES_ERR_CAPACITY;
    if (n_prompt > g.max_pos) return TILES_ERR_CAPACITY;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    float *dlog = nullptr;
    if (out_logits_host && steps > 0) {
        const size_t need = (size_t)steps * g.V;
        if (plan->logits_stage_elems < need) {
            if (plan->d_logits_stage) cudaFree(plan->d_logits_stage);
            plan->d_logits_stage = nullptr;
            plan->logits_stage_elems = 0;
            if (cudaMalloc(&plan->d_logits_stage, need * 4) != cudaSuccess) return TILES_ERR_CUDA;
            plan->logits_stage_elems = need;
        }
        dlog = plan->d_logits_stage;
    }
    if (cudaMemcpyAsync(plan->d_prompt_stage, prompt_host, (size_t)n_prompt * 4, cudaMemcpyHostToDevice, cs) !=
        cudaSuccess)
        return TILES_ERR_CUDA;
    tiles_status_t st = tiles_decode(plan, k_cache, v_cache, plan->d_prompt_stage, n_prompt, start_pos, n_new,
                                     stream, plan->d_tokens_stage, dlog);
    if (st != TILES_OK) return st;
    if (n_new > 0 && cudaMemcpyAsync(out_tokens_host, plan->d_tokens_stage, (size_t)n_new * 4,
                                     cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return TILES_ERR_CUDA;
    if (dlog && cudaMemcpyAsync(out_logits_host, dlog, (size_t)steps * g.V * 4, cudaMemcpyDeviceToHost, cs) !=
                    cudaSuccess)
        return TILES_ERR_CUDA;
    return tiles_status(plan, stream);
}

tiles_status_t tiles_quantize_rows_int8(const void *w_bf16, int32_t rows, int32_t cols, void *codes,
                                        float *scales, void *stream) {
    if (rows < 0 || cols < 1 || (rows > 0 && (!w_bf16 || !codes || !scales))) return TILES_ERR_INVALID_ARG;
    const cudaError_t e = quantize_rows_launch(w_bf16, rows, cols, codes, scales, 1, 0, 0,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TILES_OK : TILES_ERR_CUDA;
}

tiles_status_t tiles_kv8_get_layout(const tiles_model_desc *desc, tiles_kv8_layout *out) {
    if (!desc || !out || desc->n_layers < 1 || desc->n_kv_heads < 1 || desc->max_pos < 1 || desc->head_dim < 1)
        return TILES_ERR_INVALID_ARG;
    kv8_layout_of(desc->n_layers * desc->n_kv_heads, desc->max_pos, desc->head_dim, out);
    return TILES_OK;
}

tiles_status_t tiles_kv8_from_bf16(const tiles_model_desc *desc, const void *k_bf16, const void *v_bf16,
                                   int32_t n_pos, void *k8, void *v8, void *stream) {
    if (!desc || !k_bf16 || !v_bf16 || !k8 || !v8 || desc->n_layers < 1 || desc->n_kv_heads < 1 ||
        desc->max_pos < 1 || n_pos < 0 || n_pos > desc->max_pos || !aligned16(k8) || !aligned16(v8))
        return TILES_ERR_INVALID_ARG;
    if (desc->head_dim != 64 && desc->head_dim != 128) return TILES_ERR_UNSUPPORTED;
    tiles_kv8_layout lay;
    const int Z = desc->n_layers * desc->n_kv_heads, d = desc->head_dim;
    kv8_layout_of(Z, desc->max_pos, d, &lay);
    char *kb = static_cast<char *>(k8), *vb = static_cast<char *>(v8);
    const cudaError_t e = kv8_from_bf16_launch(
        static_cast<const uint16_t *>(k_bf16), static_cast<const uint16_t *>(v_bf16), Z, desc->max_pos,
        lay.pos_stride, d, n_pos, reinterpret_cast<int8_t *>(kb), reinterpret_cast<float *>(kb + lay.k_scale_off),
        reinterpret_cast<float *>(kb + lay.k_mu_off), reinterpret_cast<int8_t *>(vb),
        reinterpret_cast<float *>(vb + lay.v_scale_off), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TILES_OK : TILES_ERR_CUDA;
}

tiles_status_t tiles_copy_bw(void *dst, const void *src, size_t bytes, int32_t n_ctas, void *stream) {
    if (!dst || !src || bytes % 16 || !aligned16(dst) || !aligned16(src) || n_ctas < 0) return TILES_ERR_INVALID_ARG;
    if (bytes == 0) return TILES_OK;
    if (n_ctas == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TILES_ERR_CUDA;
        n_ctas = 2 * sms;
    }
    return copy_launch(dst, src, bytes, n_ctas, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TILES_OK
               : TILES_ERR_CUDA;
}

tiles_status_t tiles_barrier_cost(int32_t n_ctas, int32_t rounds, double *ns_per_barrier) {
    if (!ns_per_barrier || rounds < 1 || n_ctas < 0) return TILES_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TILES_ERR_CUDA;
    if (n_ctas == 0) n_ctas = sms;
    if (n_ctas > sms) return TILES_ERR_INVALID_ARG;
    uint32_t *buf = nullptr;
    if (cudaMalloc(&buf, 64) != cudaSuccess) return TILES_ERR_CUDA;
    tiles_status_t st = TILES_OK;
    unsigned long long elapsed = 0;
    uint32_t status = 0;
    if (cudaMemset(buf, 0, 64) != cudaSuccess ||
        barrier_launch(buf, rounds, reinterpret_cast<unsigned long long *>(buf + 8), buf + 4, n_ctas, 0) !=
            cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&elapsed, buf + 8, 8, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(&status, buf + 4, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = TILES_ERR_CUDA;
    else if (status)
        st = TILES_ERR_TIMEOUT;
    cudaFree(buf);
    if (st == TILES_OK) *ns_per_barrier = (double)elapsed / rounds;
    return st;
}

}  // extern "C"

namespace tiles {
bool encode_bf16_2d(TensorMap *out, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows}, ones[2] = {1, 1};
    CUtensorMap m;
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::memcpy(out, &m, sizeof m);
    return true;
}
}  // namespace tiles

// ---------------------------------------------------------------------------
// Decode without any allocation: the per-call working memory of the kernel
// (q/k/v, split partials, attention output, residual, FFN activation, argmax
// keys, phase counters, split arrivals) lives in one file-scope device array
// instead of the plan's own buffers. For callers that must not allocate device
// memory at the point of the call. The plan's tables, weights and status word
// are still the plan's.

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB, held by every GPU that loads the library
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices];  // device address of g_noalloc_scratch, per device


// Device address of the array on `dev` (current device); looked up once per device.
tiles_status_t noalloc_scratch(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return TILES_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return TILES_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = reinterpret_cast<unsigned char *>(g_noalloc_ptr[dev]);
    return TILES_OK;
}

}  // namespace

extern "C" tiles_status_t tiles_decode_noalloc(tiles_plan_t plan, void *k_cache, void *v_cache,
                                               const int32_t *prompt, int32_t n_prompt, int32_t start_pos,
                                               int32_t n_new, void *stream, int32_t *out_tokens,
                                               float *out_logits) {
    if (!plan || !k_cache || !v_cache || !prompt || n_prompt < 1 || n_new < 0 || start_pos < 0)
        return TILES_ERR_INVALID_ARG;
    if (n_new > 0 && !out_tokens) return TILES_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return TILES_ERR_INVALID_ARG;
    const Geom &g = plan->sched.geom;
    // the array holds the sync block (zeroed per launch): keys, counters and
    // every tagged activation
    const size_t need = plan->sync_bytes;
    if (need > kNoAllocScratchBytes) return TILES_ERR_CAPACITY;
    const long long steps = (long long)n_prompt - 1 + n_new;
    if (steps == 0) return TILES_OK;
    if ((long long)start_pos + steps > g.max_pos) return TILES_ERR_CAPACITY;
    tiles_status_t st = plan_check_device(plan);
    if (st != TILES_OK) return st;
    unsigned char *base = nullptr;
    if ((st = noalloc_scratch(plan->device, &base)) != TILES_OK) return st;
    KernelParams p = plan->base;
    place_sync_block(plan->sched, base, &p);
    if ((st = bind_caches(g, k_cache, v_cache, &p)) != TILES_OK) return st;
    p.prompt = prompt;
    p.n_prompt = n_prompt;
    p.out_tokens = out_tokens;
    p.out_logits = out_logits;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    for (long long s0 = 0; s0 < steps; s0 += kMaxStepsPerLaunch) {
        const int n = (int)(steps - s0 < kMaxStepsPerLaunch ? steps - s0 : kMaxStepsPerLaunch);
        p.step0 = (int)s0;
        p.pos0 = start_pos + (int)s0;
        p.n_steps = n;
        // the array keeps the previous call's contents: the counters and keys must start at zero
        cudaError_t e = cudaMemsetAsync(base, 0, plan->sync_bytes, cs);
        if (e == cudaSuccess) e = megakernel_launch(p, plan->sched.n_ctas, g.smem_bytes, cs);
        if (e != cudaSuccess) return TILES_ERR_CUDA;
    }
    return TILES_OK;
}

// Offline planner and validator (host only, no CUDA calls).
//
// Builds the tile graph of one decode step, assigns every tile to one of the
// persistent worker CTAs so that the bytes each CTA streams stay balanced,
// orders the tiles into waves (one grid barrier per phase) or dependency-
// counter chains, and validates the result before anything runs on the GPU.
// Source: "Tiles: Scheduling LLM Decoding as a Graph of Tiles", intro (tiles
// are output-row ranges with their fused work; a planner assigns every tile to
// a fixed worker, balances the bytes each worker streams, groups tiles into
// waves separated by grid barriers; the whole schedule is validated before
// launch) and the Hazy-megakernel paragraph (start work once its inputs are
// ready: the dependency-counter variant).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "tiles_internal.h"

namespace tiles {

tiles_plan_opts default_opts() {
    tiles_plan_opts o;
    std::memset(&o, 0, sizeof(o));
    o.scheduler = TILES_SCHED_FLAGS;
    return o;
}

static bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

static int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Attention scratch in the vec region: new k and v [d] bf16, per-warp states
// [G][4 + d] f32, q as bf16 [G][d + 8], and the INT8 cache's new key and
// value codes [d] with their two scales.
static int attn_vec_bytes(int G, int d) {
    return 2 * d * 2 + kConsumerWarps * G * (kPartialPad + d) * 4 + G * (d + 8) * 2 + 2 * d + 8;
}

tiles_status_t resolve_geom(const tiles_model_desc &d, const tiles_plan_opts &o, int n_ctas,
                            int smem_limit, Geom *g, std::string *why) {
    auto fail = [&](tiles_status_t st, const char *msg) {
        if (why) *why = msg;
        return st;
    };
    if (d.n_layers < 1 || d.hidden < 8 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.ffn < 8 ||
        d.vocab < 1 || d.max_pos < 1 || d.head_dim < 1)
        return fail(TILES_ERR_INVALID_ARG, "non-positive model dimension");
    if (d.tied_embeddings != 1) return fail(TILES_ERR_UNSUPPORTED, "embeddings must be tied");
    if (d.head_dim != 64 && d.head_dim != 128)
        return fail(TILES_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (d.n_q_heads % d.n_kv_heads) return fail(TILES_ERR_UNSUPPORTED, "n_q_heads % n_kv_heads");
    int G = d.n_q_heads / d.n_kv_heads;
    if (!pow2(G) || G > 8) return fail(TILES_ERR_UNSUPPORTED, "GQA group must be 1, 2, 4 or 8");
    if (d.hidden % 8 || d.ffn % 8) return fail(TILES_ERR_UNSUPPORTED, "hidden, ffn multiples of 8");
    if (d.hidden > 8192) return fail(TILES_ERR_UNSUPPORTED, "hidden above 8192");
    if (d.qk_norm != 0 && d.qk_norm != 1) return fail(TILES_ERR_INVALID_ARG, "qk_norm 0/1");
    if (d.rope_scaling != 0 && d.rope_scaling != 1)
        return fail(TILES_ERR_INVALID_ARG, "rope_scaling 0/1");
    if (!(d.rope_theta > 1.0)) return fail(TILES_ERR_INVALID_ARG, "rope_theta");
    if (!(d.rms_eps >= 0.0f)) return fail(TILES_ERR_INVALID_ARG, "rms_eps");
    if (d.rope_scaling == 1 && (!(d.rs_factor > 0) || !(d.rs_high > d.rs_low) ||
                                !(d.rs_low > 0) || d.rs_orig_max < 1))
        return fail(TILES_ERR_INVALID_ARG, "llama3 scaling parameters");
    if ((long long)d.n_q_heads * d.head_dim > 65536 || d.hidden > 65536 || d.ffn > 65536)
        return fail(TILES_ERR_UNSUPPORTED, "dimension too large");
    if (n_ctas < 1 || n_ctas > 4096) return fail(TILES_ERR_INVALID_ARG, "n_ctas");
    if (o.flags & ~(uint32_t)TILES_FLAG_INJECT_STALL) return fail(TILES_ERR_INVALID_ARG, "unknown flag bits");
    if (o.scheduler != TILES_SCHED_WAVES && o.scheduler != TILES_SCHED_COUNTERS &&
        o.scheduler != TILES_SCHED_FLAGS)
        return fail(TILES_ERR_INVALID_ARG, "scheduler");
    // 16-bit activation tags: 1 + 6 * (64 steps * layers) must stay below 2^16
    if (d.n_layers > 170) return fail(TILES_ERR_UNSUPPORTED, "more than 170 layers");

    Geom &G_ = *g;
    std::memset(&G_, 0, sizeof(G_));
    G_.L = d.n_layers;
    G_.H = d.hidden;
    G_.nq = d.n_q_heads;
    G_.nkv = d.n_kv_heads;
    G_.d = d.head_dim;
    G_.F = d.ffn;
    G_.V = d.vocab;
    G_.max_pos = d.max_pos;
    G_.G = G;
    G_.qd = d.n_q_heads * d.head_dim;
    G_.kvd = d.n_kv_heads * d.head_dim;
    G_.qkv_rows = G_.qd + 2 * G_.kvd;
    if (o.weight_format != TILES_WEIGHTS_BF16 && o.weight_format != TILES_WEIGHTS_INT8)
        return fail(TILES_ERR_INVALID_ARG, "weight_format");
    G_.wbytes = o.weight_format == TILES_WEIGHTS_INT8 ? 1 : 2;
    // INT8 rows are reduced in 16-code pieces (and copied in 16-byte units)
    if (G_.wbytes == 1 && (G_.H % 16 || G_.F % 16 || G_.qd % 16))
        return fail(TILES_ERR_UNSUPPORTED, "INT8 weights need hidden, ffn and q width multiples of 16");

    // slot: large enough for one row of every GEMV (two for gate/up). Each
    // slot has one owning consumer warp, so the default ring is one slot per
    // warp of 16 KB, or of two gate/up row pairs or the largest row if either
    // is larger: a chunk holds its slot while one warp reduces it, and smaller
    // chunks turn the ring over faster, but the gate/up stream (the most
    // bytes) must not be left one pair per chunk. Measured on GB300: Llama-1B
    // shape, 8 x 16 KB beat 6 x 32 KB by 6 % and 12 x 16 KB (uneven
    // ownership) by 2 %; Qwen3-4B shape (19 KB down rows, 10 KB gate/up
    // pairs), 8 x 20 KB slots (two pairs a chunk) beat 8 x 19 KB (one) by 17 %.
    if (o.kv_format != TILES_KV_BF16 && o.kv_format != TILES_KV_INT8)
        return fail(TILES_ERR_INVALID_ARG, "kv_format");
    G_.kv8 = o.kv_format == TILES_KV_INT8 ? 1 : 0;
    G_.kv_mp = round_up(G_.max_pos, 16);
    const int wb = G_.wbytes;
    // an INT8 KV chunk (codes of 8 KB of keys and 8 KB of values, and their
    // scales) fills one slot
    int need = std::max({wb * G_.H, wb * G_.qd, wb * G_.F, 2 * wb * G_.H, G_.kv8 ? kv8_chunk_bytes(G_.d) : 0});
    // `chain`: the chunk budget of the Q/K/V and O-projection GEMVs and of a
    // BF16 KV block, whose chunks sit on the layer's dependency chain.
    const int chain = o.slot_bytes > 0 ? o.slot_bytes : round_up(std::max({need, 16384, 4 * wb * G_.H}), 1024);
    if (chain % 1024 || chain < need) return fail(TILES_ERR_INVALID_ARG, "slot_bytes too small or not a multiple of 1024");
    // Rows per chunk: as many as fill the op's budget (`chain` for Q/K/V and
    // the O-projection, the slot for the rest). INT8 layer GEMVs are capped so
    // that a CTA's share of rows splits into at least one chunk per consumer
    // warp: a 16 KB INT8 chunk holds twice the weights of a BF16 one, and in
    // the short, latency-bound layer phases one warp's chunk arithmetic sets
    // the pace (GB300: Llama-1B shape 1547 -> 1682 tok/s, Qwen3-0.6B shape
    // 1049 -> 1273; the same cap on BF16 measured neutral, so BF16 keeps full
    // chunks). The LM head streams far more rows than warps and stays full.
    auto rpc = [&](int in, int mats, int rows, int budget) {
        const int full = std::min(kMaxRowsPerChunk, budget / (in * G_.wbytes * mats));
        if (G_.wbytes != 1 || rows <= 0) return full;
        const int per_cta = ceil_div(rows, n_ctas);
        return std::max(1, std::min(full, ceil_div(per_cta, kConsumerWarps)));
    };
    G_.rpc_qkv = rpc(G_.H, 1, G_.qkv_rows, chain);
    G_.rpc_o = rpc(G_.qd, 1, G_.H, chain);
    // KV block: whole 16-position MMA blocks (whole 32-position rounds from 32
    // on), at most one TMA box (256 rows)
    int kb = chain / (2 * G_.d * 2);
    kb = kb >= 32 ? kb / 32 * 32 : kb / 16 * 16;
    kb = std::min(kb, 256);
    if (G_.kv8) kb = kv8_block(G_.d);
    if (kb < 16) return fail(TILES_ERR_UNSUPPORTED, "slot too small for 16 KV positions");
    G_.kv_block = kb;
    int nb_max = ceil_div(G_.max_pos, kb);
    // default: one KV block per split at the longest context, at most one split
    // per CTA and KV head. Each attention tile merges a 1/S slice of its head,
    // so the merge shrinks as S grows (Llama-1B shape at 1,087 positions,
    // 64-position blocks: S = 17 ran 3 % faster than S = 9 and 6 % faster than 6).
    int splits = o.kv_splits > 0 ? o.kv_splits : std::max(1, std::min(nb_max, n_ctas / G_.nkv));
    if (splits < 1 || splits > 256) return fail(TILES_ERR_INVALID_ARG, "kv_splits");
    G_.kv_splits = splits;
    // the tensor-core owner form (and its kernel instance) only where a split
    // can hold kConsumerWarps chunks: short-context plans run kernels without
    // it, whose registers it would otherwise crowd (measured 2.5 % on the
    // Llama-1B shape at 1,023 positions)
    G_.attn_mma = (ceil_div(nb_max, splits) >= kConsumerWarps && kb % (2048 / G_.d) == 0) ? 1 : 0;
    if (G_.kv8) G_.attn_mma = 1;  // the INT8 cache has only the tensor-core form

    // an attention tile merges a 1/S slice of its KV head's G d outputs,
    // staging (m, l, o) of every (output, split) pair (3 floats each) and a
    // weight per (q head of the slice, split)
    const int per = ceil_div(G * G_.d, splits);
    const int merge_bytes = per * splits * 12 + (ceil_div(per, G_.d) + 1) * splits * 4;
    int vec = std::max({2 * G_.H, 2 * G_.qd, 2 * G_.F, attn_vec_bytes(G, G_.d), merge_bytes});
    // residual rows of an O-proj / down tile follow (a tile has at most H rows)
    G_.res_off = round_up(vec, 16);
    G_.vec_bytes = round_up(G_.res_off + 2 * G_.H, 128);
    int slot = chain;
    if (o.slot_bytes <= 0 && o.ring_slots <= 0) {
        // While the chain runs the ring fills with the layer's gate/up rows, and
        // HBM idles once it is full. So the default slot grows to the largest
        // whole number of gate/up pairs with which eight slots still fit the
        // shared memory and a CTA's gate/up share still spans two ring laps;
        // the chain's GEMVs keep `chain`-sized chunks, since fewer, longer
        // chunks there lengthen the chain. GB300, Llama-1B shape: 8 x 24 KB
        // slots (three pairs) 1542 tok/s against 1507-1522 with 16 KB; without
        // the chain budget 1493; Qwen3-0.6B shape with 24 KB slots (six pairs,
        // four chunks a CTA) 1281 against 1337-1344.
        const int pair = 2 * wb * G_.H;
        for (int k = ceil_div(G_.F, n_ctas) / (2 * kConsumerWarps); k >= 1; --k) {
            const int cand = round_up(k * pair, 1024);
            if (cand <= chain) break;
            if (kCtlBytes + kConsumerWarps * cand + G_.vec_bytes <= smem_limit) {
                slot = cand;
                break;
            }
        }
    }
    G_.slot_bytes = slot;
    G_.rpc_gateup = rpc(G_.H, 2, G_.F, slot);
    G_.rpc_down = rpc(G_.F, 1, G_.H, slot);
    G_.rpc_lm = rpc(G_.H, 1, 0, slot);
    int avail = smem_limit - kCtlBytes - G_.vec_bytes;
    int slots = o.ring_slots > 0 ? o.ring_slots : std::min(kConsumerWarps, avail / slot);
    if (slots < 2 || slots > kMaxSlots) return fail(TILES_ERR_UNSUPPORTED, "ring needs 2..32 slots");
    G_.ring_slots = slots;
    G_.smem_bytes = kCtlBytes + slots * slot + G_.vec_bytes;
    if (G_.smem_bytes > smem_limit) return fail(TILES_ERR_UNSUPPORTED, "shared memory exceeds the limit");
    return TILES_OK;
}

namespace {

struct Assign {
    int cta;
    uint32_t begin, end;
};

// Contiguous row ranges, one per CTA, sized so cumulative streamed bytes stay
// balanced: each CTA gets floor(R/N) rows and the R mod N extra rows go to the
// CTAs that have streamed least so far (ties to the lower index).
std::vector<Assign> assign_rows(int R, long long row_bytes, int N, std::vector<long long> &cum) {
    std::vector<int> cnt(N, R / N);
    int extra = R % N;
    if (extra) {
        std::vector<int> order(N);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int b) { return cum[a] < cum[b]; });
        for (int i = 0; i < extra; ++i) cnt[order[i]] += 1;
    }
    std::vector<Assign> out;
    uint32_t r = 0;
    for (int c = 0; c < N; ++c) {
        if (cnt[c] == 0) continue;
        out.push_back({c, r, r + (uint32_t)cnt[c]});
        r += cnt[c];
        cum[c] += cnt[c] * row_bytes;
    }
    return out;
}

// Single items (attention splits, combine heads) to the least-loaded CTAs,
// consecutive items merged when they land on the same CTA.
// Attention items -> CTAs: every CTA gets at most one contiguous range of
// items (so one attention task per layer). An attention task computes all its
// partials before merging, and a merge waits for every split of its head: a
// CTA holding two separate tasks would compute the second task's partials
// only after the first task's merge, delaying every merge of that head (or,
// with two splits of one head, waiting on itself until the timeout). The
// least-loaded CTAs so far take the items: with no more items than CTAs one
// each, the heaviest item to the least-loaded CTA; otherwise contiguous ranges,
// the first n_items mod N of them one item longer.
// `allowed` (ascending CTA indices) restricts the takers; empty = every CTA.
std::vector<Assign> assign_items(int n_items, const std::vector<long long> &item_bytes, int N,
                                 std::vector<long long> &cum, const std::vector<int> &allowed) {
    std::vector<int> order = allowed;
    if (order.empty()) {
        order.resize(N);
        for (int c = 0; c < N; ++c) order[c] = c;
    }
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cum[a] < cum[b]; });
    if (n_items <= (int)order.size()) {
        std::vector<int> items(n_items);
        for (int i = 0; i < n_items; ++i) items[i] = i;
        std::stable_sort(items.begin(), items.end(),
                         [&](int a, int b) { return item_bytes[a] > item_bytes[b]; });
        std::vector<Assign> out;
        for (int k = 0; k < n_items; ++k) {
            out.push_back({order[k], (uint32_t)items[k], (uint32_t)items[k] + 1});
            cum[order[k]] += item_bytes[items[k]];
        }
        std::sort(out.begin(), out.end(), [](const Assign &x, const Assign &y) { return x.begin < y.begin; });
        return out;
    }
    const int takers = (int)order.size();
    std::vector<int> ctas(order.begin(), order.begin() + takers);
    std::sort(ctas.begin(), ctas.end());  // ranges in CTA order
    std::vector<Assign> out;
    int it = 0;
    for (int k = 0; k < takers; ++k) {
        const int n = n_items / takers + (k < n_items % takers ? 1 : 0);
        Assign a{ctas[k], (uint32_t)it, (uint32_t)(it + n)};
        for (int i = it; i < it + n; ++i) cum[ctas[k]] += item_bytes[i];
        it += n;
        out.push_back(a);
    }
    return out;
}

// CTAs that may hold attention items. Under tag-carrying activations an
// attention CTA orders its K/V writes before the next step's copies through
// its own LM-head signal, so it must hold LM-head rows. With at least one
// vocabulary row per CTA every CTA does (no restriction). With fewer rows the
// attention items of every layer go to V CTAs spread evenly over the grid,
// and each of them takes one LM-head row.
std::vector<int> attention_ctas(const Geom &g, int N) {
    std::vector<int> a;
    if (g.V >= N) return a;
    for (int i = 0; i < g.V; ++i) a.push_back((int)((long long)i * N / g.V));
    return a;
}

}  // namespace

tiles_status_t build_schedule(const tiles_model_desc &d, const tiles_plan_opts &o, int N,
                              int smem_limit, tiles_schedule_s *s, std::string *why) {
    tiles_status_t st = resolve_geom(d, o, N, smem_limit, &s->geom, why);
    if (st != TILES_OK) return st;
    const Geom &g = s->geom;
    s->desc = d;
    s->opts = o;
    s->n_ctas = N;
    s->scheduler = o.scheduler;
    const int PPS = phases_per_step(g);

    // per phase, the (cta, range) tasks
    std::vector<std::vector<Assign>> phase_tasks(PPS);
    std::vector<int> phase_op(PPS), phase_layer(PPS);
    std::vector<long long> cum(N, 0);
    const std::vector<int> attn_ctas = attention_ctas(g, N);
    // attention bytes for balancing: split sizes at the largest position
    for (int l = 0; l <= g.L; ++l) {
        for (int k = 0; k < (l < g.L ? kPhaseKinds : 1); ++k) {
            int kind = l < g.L ? k : 6;
            int phi = phase_index(g, l < g.L ? l : 0, kind);
            static const int ops[7] = {TILES_OP_QKV,  TILES_OP_ATTN,   TILES_OP_COMBINE,
                                       TILES_OP_OPROJ, TILES_OP_GATEUP, TILES_OP_DOWN,
                                       TILES_OP_LMHEAD};
            int op = ops[kind];
            phase_op[phi] = op;
            phase_layer[phi] = l < g.L ? l : 0;
            const long long row_bytes = (long long)op_in_dim(g, op) * g.wbytes * op_mats(op);
            if (op == TILES_OP_LMHEAD && !attn_ctas.empty()) {
                // one vocabulary row to each attention CTA, in CTA (= row) order
                for (int i = 0; i < g.V; ++i) {
                    phase_tasks[phi].push_back({attn_ctas[i], (uint32_t)i, (uint32_t)i + 1});
                    cum[attn_ctas[i]] += row_bytes;
                }
            } else if (op_is_gemv(op)) {
                phase_tasks[phi] = assign_rows(op_extent(g, op), row_bytes, N, cum);
            } else if (op == TILES_OP_ATTN) {
                int n = op_extent(g, op);
                std::vector<long long> b(n);
                for (int it = 0; it < n; ++it) {
                    tiles_task t{};
                    t.op = TILES_OP_ATTN;
                    t.begin = it;
                    t.end = it + 1;
                    b[it] = task_bytes(g, t, g.max_pos - 1);
                }
                phase_tasks[phi] = assign_items(n, b, N, cum, attn_ctas);
            }
            // the combine phase stays empty: the last split tile of each KV head
            // merges the partials inside the attention phase
        }
    }

    // counters and waits
    std::vector<std::vector<tiles_task>> per_cta(N);
    std::vector<int> ord(PPS, 0);  // index among non-empty phases
    int n_nonempty = 0;
    for (int phi = 0; phi < PPS; ++phi) {
        ord[phi] = n_nonempty;
        if (!phase_tasks[phi].empty()) ++n_nonempty;
    }
    if (o.scheduler == TILES_SCHED_WAVES) {
        s->n_counters = 1;
        for (int phi = 0; phi < PPS; ++phi) {
            if (phase_tasks[phi].empty()) continue;
            std::vector<bool> has(N, false);
            std::vector<int> last(N, -1);
            for (size_t k = 0; k < phase_tasks[phi].size(); ++k) last[phase_tasks[phi][k].cta] = (int)k;
            for (size_t k = 0; k < phase_tasks[phi].size(); ++k) {
                const Assign &a = phase_tasks[phi][k];
                tiles_task t{};
                t.op = (uint8_t)phase_op[phi];
                t.phase_kind = (uint8_t)phase_of_op(phase_op[phi]);
                t.layer = (uint16_t)phase_layer[phi];
                t.begin = a.begin;
                t.end = a.end;
                t.wait_ctr = 0;
                // one arrival per CTA and phase, after its last task of the phase
                t.signal_ctr = last[a.cta] == (int)k ? 0 : TILES_NO_COUNTER;
                t.wait_mul = (uint32_t)(N * n_nonempty);
                t.wait_add = (uint32_t)(N * ord[phi]);
                has[a.cta] = true;
                per_cta[a.cta].push_back(t);
            }
            for (int c = 0; c < N; ++c) {
                if (has[c]) continue;
                tiles_task t{};
                t.op = TILES_OP_SYNC;
                t.phase_kind = (uint8_t)phase_of_op(phase_op[phi]);
                t.layer = (uint16_t)phase_layer[phi];
                t.wait_ctr = 0;
                t.signal_ctr = 0;
                t.wait_mul = (uint32_t)(N * n_nonempty);
                t.wait_add = (uint32_t)(N * ord[phi]);
                per_cta[c].push_back(t);
            }
        }
        s->final_ctr = 0;
        s->final_mul = (uint32_t)(N * n_nonempty);
    } else {
        s->n_counters = PPS;
        // previous non-empty phase, cyclically (phase 0 depends on the last of the step before)
        std::vector<int> prev(PPS, -1);
        int last_nonempty = -1;
        for (int phi = PPS - 1; phi >= 0 && last_nonempty < 0; --phi)
            if (!phase_tasks[phi].empty()) last_nonempty = phi;
        int p = last_nonempty;
        for (int phi = 0; phi < PPS; ++phi) {
            prev[phi] = p;
            if (!phase_tasks[phi].empty()) p = phi;
        }
        // signals per step: one per task
        auto per_step = [&](int phi) -> uint32_t {
            return phi < 0 ? 0u : (uint32_t)phase_tasks[phi].size();
        };
        for (int phi = 0; phi < PPS; ++phi) {
            int pp = prev[phi];
            uint32_t npp = per_step(pp);
            for (auto &a : phase_tasks[phi]) {
                tiles_task t{};
                t.op = (uint8_t)phase_op[phi];
                t.phase_kind = (uint8_t)phase_of_op(phase_op[phi]);
                t.layer = (uint16_t)phase_layer[phi];
                t.begin = a.begin;
                t.end = a.end;
                t.signal_ctr = (uint16_t)phi;
                t.wait_ctr = (uint16_t)pp;
                t.wait_mul = npp;
                t.wait_add = pp < phi ? npp : 0;  // same step, or the step before
                if (o.scheduler == TILES_SCHED_FLAGS) {
                    // tagged inputs need no counter: only the first Q/K/V tile of a
                    // step (reads the sampled token) waits, and only the LM head signals
                    const int op = phase_op[phi];
                    const bool waits = op == TILES_OP_QKV && phase_layer[phi] == 0;
                    const bool signals = op == TILES_OP_LMHEAD;
                    if (!waits) {
                        t.wait_ctr = TILES_NO_COUNTER;
                        t.wait_mul = t.wait_add = 0;
                    }
                    if (!signals) t.signal_ctr = TILES_NO_COUNTER;
                }
                per_cta[a.cta].push_back(t);
            }
        }
        s->final_ctr = last_nonempty;
        s->final_mul = per_step(last_nonempty);
    }
    s->tasks.clear();
    s->offsets.assign(N + 1, 0);
    for (int c = 0; c < N; ++c) {
        s->offsets[c] = (int32_t)s->tasks.size();
        s->tasks.insert(s->tasks.end(), per_cta[c].begin(), per_cta[c].end());
    }
    s->offsets[N] = (int32_t)s->tasks.size();
    return TILES_OK;
}

tiles_status_t validate_schedule(const tiles_schedule_s &s, std::string *why) {
    char buf[256];
    auto fail = [&](const char *msg) {
        if (why) *why = msg;
        return TILES_ERR_PLAN_INVALID;
    };
    const Geom &g = s.geom;
    const int N = s.n_ctas, PPS = phases_per_step(g);
    if ((int)s.offsets.size() != N + 1 || s.offsets[0] != 0 ||
        s.offsets[N] != (int32_t)s.tasks.size())
        return fail("task offsets inconsistent");
    // geometry: every copy is a whole number of 16-byte units into 128-byte aligned slots
    if (g.slot_bytes % 1024 || g.ring_slots < 2 || g.ring_slots > kMaxSlots)
        return fail("ring geometry");
    if ((g.wbytes * g.H) % 16 || (g.wbytes * g.F) % 16 || (g.wbytes * g.qd) % 16 || (2 * g.d) % 16)
        return fail("row bytes not a multiple of 16");
    for (int op = TILES_OP_QKV; op <= TILES_OP_LMHEAD; ++op) {
        if (!op_is_gemv(op)) continue;
        int r = op_rows_per_chunk(g, op);
        if (r < 1 || (long long)r * op_in_dim(g, op) * g.wbytes * op_mats(op) > g.slot_bytes)
            return fail("rows per chunk do not fit a slot");
    }
    const long long kv_chunk = g.kv8 ? kv8_chunk_bytes(g.d) : 2LL * g.kv_block * g.d * 2;
    if (g.kv_block < 16 || g.kv_block > 256 || g.kv_block % 16 || kv_chunk > g.slot_bytes) return fail("kv block");
    if (g.attn_mma && g.kv_block % (2048 / g.d)) return fail("kv block not a whole number of tensor-core rounds");
    if (g.kv8 && (g.kv_block != kv8_block(g.d) || !g.attn_mma || g.kv_mp % 16 || g.kv_mp < g.max_pos))
        return fail("INT8 KV chunk geometry");
    if (g.smem_bytes > kSmemLimit) return fail("shared memory");
    if (s.n_counters < 1 || s.n_counters > 0xFFFE) return fail("counter count");

    // per phase coverage, per CTA order, signal accounting
    std::vector<std::vector<std::pair<uint32_t, uint32_t>>> cover(PPS);
    std::vector<int> phase_op(PPS, 0);
    std::vector<std::vector<int>> sig_by_phase(PPS, std::vector<int>(s.n_counters, 0));
    for (int c = 0; c < N; ++c) {
        int last_phi = -1;
        for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i) {
            if (i < s.offsets[c] || i >= (int)s.tasks.size()) return fail("task index");
            const tiles_task &t = s.tasks[i];
            if (t.op < TILES_OP_QKV || t.op > TILES_OP_SYNC) return fail("unknown op");
            int kind = t.op == TILES_OP_SYNC ? t.phase_kind : phase_of_op(t.op);
            if (kind < 0 || kind > 6 || t.phase_kind != kind) return fail("phase kind mismatch");
            if (kind < 6 && t.layer >= g.L) return fail("layer out of range");
            int phi = phase_index(g, kind == 6 ? 0 : t.layer, kind);
            if (phi < last_phi) return fail("tasks of a CTA out of phase order");
            last_phi = phi;
            if (t.op != TILES_OP_SYNC) {
                if (phase_op[phi] && phase_op[phi] != t.op) return fail("two ops in one phase");
                phase_op[phi] = t.op;
                if (t.begin >= t.end || t.end > (uint32_t)op_extent(g, t.op))
                    return fail("task range out of bounds");
                cover[phi].push_back({t.begin, t.end});
            }
            if (t.signal_ctr != TILES_NO_COUNTER) {
                if (t.signal_ctr >= s.n_counters) return fail("signal counter out of range");
                sig_by_phase[phi][t.signal_ctr] += 1;
            }
            if (t.wait_ctr != TILES_NO_COUNTER && t.wait_ctr >= s.n_counters)
                return fail("wait counter out of range");
        }
    }
    for (int c = 0; c < N; ++c) {
        std::vector<char> seen(g.L, 0);
        for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i) {
            const tiles_task &t = s.tasks[i];
            if (t.op != TILES_OP_ATTN) continue;
            if (seen[t.layer]) return fail("two attention tasks of one layer on one CTA (merge order)");
            seen[t.layer] = 1;
        }
    }
    for (int phi = 0; phi < PPS; ++phi) {
        auto &v = cover[phi];
        std::sort(v.begin(), v.end());
        int kind = phi == PPS - 1 ? 6 : phi % kPhaseKinds;
        static const int ops[7] = {TILES_OP_QKV,  TILES_OP_ATTN,   TILES_OP_COMBINE,
                                   TILES_OP_OPROJ, TILES_OP_GATEUP, TILES_OP_DOWN,
                                   TILES_OP_LMHEAD};
        uint32_t want = (uint32_t)op_extent(g, ops[kind]);
        uint32_t at = 0;
        for (auto &r : v) {
            if (r.first != at) {
                std::snprintf(buf, sizeof buf, "phase %d: rows/items [%u, %u) %s", phi, at,
                              r.first, r.first > at ? "not covered" : "covered twice");
                if (why) *why = buf;
                return TILES_ERR_PLAN_INVALID;
            }
            at = r.second;
        }
        if (at != want) {
            std::snprintf(buf, sizeof buf, "phase %d: covers %u of %u rows/items", phi, at, want);
            if (why) *why = buf;
            return TILES_ERR_PLAN_INVALID;
        }
    }
    // signals per step on each counter; per CTA, the counter its last task of each phase signals
    std::vector<long long> per_step(s.n_counters, 0);
    for (int phi = 0; phi < PPS; ++phi)
        for (int c = 0; c < s.n_counters; ++c) per_step[c] += sig_by_phase[phi][c];
    std::vector<int> last_sig((size_t)N * PPS, -2);  // -2: no task of the CTA in that phase
    std::vector<int> phase_ntasks(PPS, 0);
    for (int c = 0; c < N; ++c)
        for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i) {
            const tiles_task &t = s.tasks[i];
            int kind = t.op == TILES_OP_SYNC ? t.phase_kind : phase_of_op(t.op);
            int phi = phase_index(g, kind == 6 ? 0 : t.layer, kind);
            phase_ntasks[phi] += 1;
            last_sig[(size_t)c * PPS + phi] =
                t.signal_ctr == TILES_NO_COUNTER ? -1 : (int)t.signal_ctr;
        }
    for (int c = 0; c < N; ++c) {
        for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i) {
            const tiles_task &t = s.tasks[i];
            int kind = t.op == TILES_OP_SYNC ? t.phase_kind : phase_of_op(t.op);
            int phi = phase_index(g, kind == 6 ? 0 : t.layer, kind);
            if (t.wait_ctr == TILES_NO_COUNTER) {
                // only tiles whose inputs are all tagged words may skip the counters
                const bool tagged_inputs = t.op == TILES_OP_ATTN || t.op == TILES_OP_OPROJ ||
                                           t.op == TILES_OP_GATEUP || t.op == TILES_OP_DOWN ||
                                           t.op == TILES_OP_LMHEAD || (t.op == TILES_OP_QKV && t.layer > 0);
                if (s.scheduler != TILES_SCHED_FLAGS || !tagged_inputs) return fail("task without a wait");
                continue;
            }
            int ctr = t.wait_ctr;
            long long before = 0;
            for (int q = 0; q < phi; ++q) before += sig_by_phase[q][ctr];
            if ((long long)t.wait_mul != per_step[ctr])
                return fail("wait multiplier differs from the counter's signals per step");
            if ((long long)t.wait_add != before)
                return fail("wait target is not exactly the signals issued before this phase");
            // the wait must cover the nearest earlier non-empty phase (cyclically): every CTA
            // with work there signals this counter after its last task of that phase
            int prev = -1;
            for (int q = phi - 1; q >= 0 && prev < 0; --q)
                if (phase_ntasks[q]) prev = q;
            for (int q = PPS - 1; q > phi && prev < 0; --q)
                if (phase_ntasks[q]) prev = q;
            if (prev < 0) continue;
            for (int c2 = 0; c2 < N; ++c2) {
                int ls = last_sig[(size_t)c2 * PPS + prev];
                if (ls != -2 && ls != ctr)
                    return fail("wait does not cover every task of the previous phase");
            }
        }
    }
    if (s.final_ctr < 0 || s.final_ctr >= s.n_counters || (long long)s.final_mul != per_step[s.final_ctr])
        return fail("final wait");
    if (s.scheduler == TILES_SCHED_FLAGS) {
        // The K/V an attention tile writes is read by TMA in later steps, and
        // its only ordering is a release by the same CTA: its LM-head tile's
        // signal, which the first tile of the next step acquires. So every CTA
        // with attention work must also signal the LM-head counter.
        for (int c = 0; c < N; ++c) {
            bool attn = false, lm = false;
            for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i) {
                const tiles_task &t = s.tasks[i];
                attn |= t.op == TILES_OP_ATTN;
                lm |= t.op == TILES_OP_LMHEAD && t.signal_ctr != TILES_NO_COUNTER;
            }
            if (attn && !lm) return fail("an attention CTA does not signal the LM head (K/V ordering)");
        }
    }
    return TILES_OK;
}

}  // namespace tiles

using namespace tiles;

extern "C" {

tiles_status_t tiles_schedule_build(const tiles_model_desc *desc, const tiles_plan_opts *opts,
                                    int32_t n_ctas, tiles_schedule_t *out) {
    if (!desc || !out) return TILES_ERR_INVALID_ARG;
    *out = nullptr;
    tiles_plan_opts o = opts ? *opts : default_opts();
    auto *s = new tiles_schedule_s();
    std::string why;
    tiles_status_t st = build_schedule(*desc, o, n_ctas, kSmemLimit, s, &why);
    if (st != TILES_OK) {
        delete s;
        return st;
    }
    *out = s;
    return TILES_OK;
}

tiles_status_t tiles_schedule_validate(tiles_schedule_t sched, char *why, size_t why_len) {
    if (!sched) return TILES_ERR_INVALID_ARG;
    std::string w;
    tiles_status_t st = validate_schedule(*sched, &w);
    if (why && why_len) {
        std::snprintf(why, why_len, "%s", st == TILES_OK ? "ok" : w.c_str());
    }
    return st;
}

tiles_status_t tiles_schedule_tasks(tiles_schedule_t sched, tiles_task **tasks, int32_t *n_tasks,
                                    const int32_t **offsets, int32_t *n_ctas) {
    if (!sched || !tasks || !n_tasks || !offsets || !n_ctas) return TILES_ERR_INVALID_ARG;
    *tasks = sched->tasks.data();
    *n_tasks = (int32_t)sched->tasks.size();
    *offsets = sched->offsets.data();
    *n_ctas = sched->n_ctas;
    return TILES_OK;
}

tiles_status_t tiles_schedule_cta_bytes(tiles_schedule_t sched, int32_t pos, int64_t *bytes) {
    if (!sched || !bytes || pos < 0 || pos >= sched->geom.max_pos) return TILES_ERR_INVALID_ARG;
    for (int c = 0; c < sched->n_ctas; ++c) {
        long long b = 0;
        for (int i = sched->offsets[c]; i < sched->offsets[c + 1]; ++i)
            b += task_bytes(sched->geom, sched->tasks[i], pos);
        bytes[c] = b;
    }
    return TILES_OK;
}

tiles_status_t tiles_schedule_get_info(tiles_schedule_t sched, tiles_plan_info *info) {
    if (!sched || !info) return TILES_ERR_INVALID_ARG;
    const tiles_schedule_s &s = *sched;
    const Geom &g = s.geom;
    std::memset(info, 0, sizeof(*info));
    info->n_ctas = s.n_ctas;
    info->threads_per_cta = kThreads;
    info->smem_bytes = g.smem_bytes;
    info->slot_bytes = g.slot_bytes;
    info->ring_slots = g.ring_slots;
    info->kv_splits = g.kv_splits;
    info->scheduler = s.scheduler;
    info->n_tasks = (int32_t)s.tasks.size();
    info->n_counters = s.n_counters;
    info->phases_per_step = phases_per_step(g);
    int mt = 0;
    for (int c = 0; c < s.n_ctas; ++c) mt = std::max(mt, s.offsets[c + 1] - s.offsets[c]);
    info->max_tasks_per_cta = mt;
    info->kv_block = g.kv_block;
    info->attn_tensor_cores = g.attn_mma;
    info->rows_per_chunk[0] = g.rpc_qkv;
    info->rows_per_chunk[1] = g.rpc_o;
    info->rows_per_chunk[2] = g.rpc_gateup;
    info->rows_per_chunk[3] = g.rpc_down;
    info->rows_per_chunk[4] = g.rpc_lm;
    info->weight_format = g.wbytes == 1 ? TILES_WEIGHTS_INT8 : TILES_WEIGHTS_BF16;
    info->kv_format = g.kv8 ? TILES_KV_INT8 : TILES_KV_BF16;
    long long tot = 0, mx = 0, mn = -1;
    for (int c = 0; c < s.n_ctas; ++c) {
        long long b = 0;
        for (int i = s.offsets[c]; i < s.offsets[c + 1]; ++i)
            if (op_is_gemv(s.tasks[i].op)) b += task_bytes(g, s.tasks[i], 0);
        tot += b;
        mx = b > mx ? b : mx;
        mn = (mn < 0 || b < mn) ? b : mn;
    }
    info->weight_bytes_per_token = tot;
    info->max_cta_bytes = mx;
    info->min_cta_bytes = mn;
    return TILES_OK;
}

void tiles_schedule_destroy(tiles_schedule_t sched) { delete sched; }

const char *tiles_status_string(tiles_status_t st) {
    switch (st) {
        case TILES_OK: return "ok";
        case TILES_ERR_INVALID_ARG: return "invalid argument";
        case TILES_ERR_UNSUPPORTED: return "unsupported model shape";
        case TILES_ERR_PLAN_INVALID: return "plan failed validation";
        case TILES_ERR_DEVICE_MISMATCH: return "plan made for another device or binary";
        case TILES_ERR_CAPACITY: return "start_pos + steps exceeds max_pos";
        case TILES_ERR_CUDA: return "CUDA runtime error";
        case TILES_ERR_TIMEOUT: return "in-kernel wait timed out";
        case TILES_ERR_DEVICE_BOUNDS: return "kernel rejected an out-of-range index";
        default: return "unknown status";
    }
}

}  // extern "C"

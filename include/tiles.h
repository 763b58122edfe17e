/*
 * tiles.h -- C ABI of the tile-scheduled persistent decoder for GB300 (sm_103a).
 *
 * The operation: batch-size-1 greedy decoding of a Llama/Qwen-style dense BF16
 * decoder in which every operator is cut into tiles (a range of output rows
 * plus the small fused work that produces them), an offline planner assigns
 * every tile to one persistent worker CTA per SM, balances the bytes each
 * worker streams and orders the tiles, and one persistent kernel executes the
 * whole schedule for a run of up to 64 tokens, with greedy selection inside
 * the kernel.  Sources: "Tiles: Scheduling LLM Decoding as a Graph of Tiles"
 * (intro; "What the code contains": the planner validates the schedule, the
 * runtime re-validates it, checks it was made for this binary and GPU, and runs
 * up to 64 tokens per cooperative launch with greedy selection in the kernel;
 * "Scope": prefill one token per step).
 *
 * Conventions for every function below:
 *   - All pointers are plain addresses. "device" means CUDA device memory of
 *     the GPU the plan was made on; "host" means ordinary host memory.
 *   - Matrices are row-major [out][in] bfloat16 (uint16 bit patterns).
 *   - The caller owns every buffer it passes in (weights, caches, prompts,
 *     outputs); they must stay valid while a plan or call uses them. A plan
 *     owns only what it allocates itself (its tables and scratch).
 *   - Functions return TILES_OK or a negative tiles_status_t and never abort
 *     the process. A NULL required pointer gives TILES_ERR_INVALID_ARG.
 *   - A plan is not thread-safe: one decode in flight per plan.
 */
#ifndef TILES_H
#define TILES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TILES_OK = 0,
    TILES_ERR_INVALID_ARG = -1,     /* bad pointer, size or option                    */
    TILES_ERR_UNSUPPORTED = -2,     /* shape outside what the kernel handles          */
    TILES_ERR_PLAN_INVALID = -3,    /* schedule failed validation                     */
    TILES_ERR_DEVICE_MISMATCH = -4, /* plan used on another GPU / SM count / binary   */
    TILES_ERR_CAPACITY = -5,        /* start_pos + steps exceeds max_pos              */
    TILES_ERR_CUDA = -6,            /* a CUDA runtime call failed                     */
    TILES_ERR_TIMEOUT = -7,         /* a bounded in-kernel wait expired               */
    TILES_ERR_DEVICE_BOUNDS = -8    /* the kernel rejected an out-of-range index      */
} tiles_status_t;

/* Model shape.  Llama-style when qk_norm == 0, Qwen3-style (per-head RMSNorm on
 * q and k before RoPE) when qk_norm == 1.  Embeddings must be tied (the LM head
 * is the embedding matrix).  RoPE pairs element j with j + head_dim/2; inverse
 * frequencies theta^(-2j/d) with optional llama3 scaling (rope_scaling == 1,
 * factor / low / high / original context), angles and tables in FP64 rounded
 * to FP32. */
typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_pos;
    int32_t qk_norm;          /* 0 or 1                                   */
    int32_t rope_scaling;     /* 0 none, 1 llama3                          */
    int32_t tied_embeddings;  /* must be 1                                */
    int32_t rs_orig_max;      /* llama3: original context length          */
    double rope_theta;
    double rs_factor, rs_low, rs_high;
    float rms_eps;            /* RMSNorm epsilon, also for the q/k norms  */
} tiles_model_desc;

/* Device pointers to one layer's weights. q_norm / k_norm are [head_dim] and
 * may be NULL when qk_norm == 0. */
typedef struct {
    const void *attn_norm;  /* [hidden]                       */
    const void *wq;         /* [n_q_heads*head_dim][hidden]   */
    const void *wk;         /* [n_kv_heads*head_dim][hidden]  */
    const void *wv;         /* [n_kv_heads*head_dim][hidden]  */
    const void *q_norm;     /* [head_dim] or NULL             */
    const void *k_norm;     /* [head_dim] or NULL             */
    const void *wo;         /* [hidden][n_q_heads*head_dim]   */
    const void *ffn_norm;   /* [hidden]                       */
    const void *w_gate;     /* [ffn][hidden]                  */
    const void *w_up;       /* [ffn][hidden]                  */
    const void *w_down;     /* [hidden][ffn]                  */
} tiles_layer_weights;

/* Device weight pointers; every pointer 16-byte aligned. `layers` itself is a
 * HOST array of n_layers entries (copied by tiles_plan_create). */
typedef struct {
    const void *embed;       /* [vocab][hidden], also the LM head */
    const void *final_norm;  /* [hidden]                          */
    const tiles_layer_weights *layers;
} tiles_weights;

/* How tiles wait for their inputs.
 *  WAVES: every phase ends in a grid barrier (a counter all CTAs arrive on).
 *  COUNTERS: a tile waits on the dependency counter of the phase it reads,
 *    which every tile of that phase increments once done.
 *  FLAGS (default): activations carry their own readiness. Each word of the
 *    residual stream, the Q/K/V projection, the split-KV partials, the
 *    attention output and the SwiGLU output holds the value and the tag of
 *    the (step, layer, phase) that wrote it, and a tile polls the words it
 *    reads until they carry the tag it expects. Only the sampled token still
 *    goes through a counter (the LM-head tiles signal it).
 * All three compute bit-identical results. */
enum { TILES_SCHED_WAVES = 0, TILES_SCHED_COUNTERS = 1, TILES_SCHED_FLAGS = 2 };

/* Weights the GEMV tiles stream. BF16: the caller's matrices (Q/K/V and
 * gate/up repacked by the plan). INT8 ("History and roadmap", "Milestones":
 * weight-only INT8 linear layers): at plan creation every GEMV matrix, the
 * tied LM head included, is quantized per output row with
 * tiles_quantize_rows_int8 into plan-owned codes and FP32 scales, and a GEMV
 * row becomes scale * sum(code * x). Activations, norms, the KV cache and the
 * embedding lookup stay BF16. INT8 needs hidden, ffn and n_q_heads * head_dim
 * to be multiples of 16. */
enum { TILES_WEIGHTS_BF16 = 0, TILES_WEIGHTS_INT8 = 1 };

/* KV cache formats. TILES_KV_BF16: the k_cache / v_cache of the decode calls
 * are BF16 [L][n_kv][max_pos][head_dim]. TILES_KV_INT8 ("History and
 * roadmap", "M8 so far": INT8 KV cache with smoothed keys; "Tried and not
 * kept": queries stay unquantized): each cached row is INT8 codes with one
 * FP32 scale, and keys are stored minus a per-(layer, KV head) channel mean
 * mu (the smoothing):
 *   key row:   x = R(k) - mu;  value row: x = R(v)   (R = the BF16 rounding)
 *   s = max_j |x_j| / 127,  c_j = x_j / s rounded to nearest even, clamped
 *   to [-127, 127] (all in FP32; an all-zero row: s = 0, codes 0).
 * Attention reads K_t = s_t c_t and V_t likewise, and never adds mu back:
 * it moves every score of a query by q . mu, which the softmax cancels.
 * mu comes from the prefill (tiles_kv8_from_bf16) and stays fixed while
 * decoding. See tiles_kv8_layout for the two buffers. */
enum { TILES_KV_BF16 = 0, TILES_KV_INT8 = 1 };

/* Planner options; pass NULL to tiles_plan_create for the defaults (shown). */
typedef struct {
    int32_t scheduler;    /* TILES_SCHED_FLAGS (default), _COUNTERS or _WAVES            */
    int32_t n_ctas;       /* 0 = one worker CTA per SM                                  */
    int32_t slot_bytes;   /* ring slot bytes, a multiple of 1024. 0 = auto: Q/K/V, O and
                           * KV-block chunks fill 16 KB (or the longest row, or two
                           * gate/up row pairs, if larger); the slot, which gate/up,
                           * down and LM-head chunks fill, grows from there to whole
                           * gate/up pairs while 8 slots fit shared memory and a CTA's
                           * gate/up rows still make 16 chunks. Nonzero: every chunk
                           * fills this size.                                         */
    int32_t ring_slots;   /* 0 = one per consumer warp (8), fewer if they do not fit;
                           * nonzero also keeps the slot at the 16 KB rule             */
    int32_t kv_splits;    /* 0 = auto: split-KV ranges per KV head                       */
    int32_t timeout_ms;   /* bound on every in-kernel wait; 0 = 2000 ms                  */
    int32_t l2_prefetch_kb; /* L2 prefetch warp: weight bytes it may run ahead of the ring, KB per CTA; <= 0 = off */
    int32_t l2_prefetch_gbs; /* its issue rate per CTA, GB/s (token bucket); <= 0 = unpaced */
    int32_t weight_format; /* TILES_WEIGHTS_BF16 (default) or TILES_WEIGHTS_INT8           */
    uint32_t flags;       /* TILES_FLAG_* bits; 0 for normal use                         */
    int32_t kv_format;    /* TILES_KV_BF16 (default) or TILES_KV_INT8                     */
} tiles_plan_opts;

/* TILES_FLAG_INJECT_STALL is a test hook for failure detection. After the
 * schedule is validated, the first tile of CTA 0 is made to wait for a
 * counter value no launch reaches. Every bounded wait of the launch then runs
 * out: the launch ends with TILES_ERR_TIMEOUT in the status word (read with
 * tiles_status) after about timeout_ms, and nothing faults. */
enum { TILES_FLAG_INJECT_STALL = 1u };

typedef struct tiles_plan_s *tiles_plan_t;

/* Builds, validates and uploads a schedule for `desc` on the current CUDA
 * device ("Tiles: Scheduling LLM Decoding as a Graph of Tiles", intro: the
 * offline planner; "What the code contains": the schedule is validated before
 * launch). Query the device (SM count, shared memory, cooperative launch,
 * occupancy of the worker kernel at the chosen shared-memory size), build the
 * tile graph, assign tiles to CTAs balancing streamed bytes, order them into
 * waves or dependency-counter chains, validate, and allocate the plan's own
 * device tables and scratch. The plan also packs its own copies of
 * [Wq; Wk; Wv] and of Wg/Wu interleaved by row (the kernel streams those, one
 * bulk copy per ring chunk); wq/wk/wv/w_gate/w_up are only read during this
 * call. With TILES_WEIGHTS_INT8 the plan holds codes of every GEMV matrix, so
 * wo and w_down are only read here too. The embedding and the norm gains (and,
 * for BF16, wo and w_down) must stay valid for the plan's lifetime. On success *out owns its
 * allocations. Errors: INVALID_ARG, UNSUPPORTED (shape), PLAN_INVALID, CUDA. */
tiles_status_t tiles_plan_create(const tiles_model_desc *desc, const tiles_weights *weights,
                                 const tiles_plan_opts *opts, tiles_plan_t *out);

/* Frees everything the plan allocated (no counterpart on the pages). NULL is
 * allowed. The caller must make sure no decode using the plan is still
 * running. */
void tiles_plan_destroy(tiles_plan_t plan);

/*
 * Greedy decoding, asynchronous on `stream` (a cudaStream_t, NULL = legacy).
 * ("Tiles: Scheduling LLM Decoding as a Graph of Tiles", intro and "What the
 * code contains": one persistent kernel runs the whole schedule for up to 64
 * tokens per cooperative launch, greedy selection inside the kernel; "Scope
 * and code release": the prompt goes one token per step.)
 *
 * Runs n_prompt - 1 + n_new steps; step s runs at position start_pos + s. Its
 * input token is prompt[s] when s < n_prompt, else the token chosen at step
 * s - 1. Steps s >= n_prompt - 1 write out_tokens[s - (n_prompt - 1)]. Every
 * step writes K and V of its position into the caches and reads positions
 * 0..start_pos + s. Steps are split into cooperative launches of <= 64.
 *
 *   k_cache, v_cache  device, [n_layers][n_kv_heads][max_pos][head_dim] bf16,
 *                     positions < start_pos already filled by the caller;
 *                     with kv_format TILES_KV_INT8, the two INT8 cache
 *                     buffers of tiles_kv8_layout (positions < start_pos
 *                     filled, e.g. by tiles_kv8_from_bf16)
 *   prompt            device, n_prompt >= 1 token ids in [0, vocab)
 *   out_tokens        device, n_new int32
 *   out_logits        device, [n_prompt - 1 + n_new][vocab] float32, or NULL
 *
 * The return value covers argument, capacity and launch errors; errors raised
 * inside the kernel (timeout, bad token id) are read by tiles_status.
 * Errors: INVALID_ARG, CAPACITY, DEVICE_MISMATCH, CUDA.
 */
tiles_status_t tiles_decode(tiles_plan_t plan, void *k_cache, void *v_cache,
                            const int32_t *prompt, int32_t n_prompt, int32_t start_pos,
                            int32_t n_new, void *stream, int32_t *out_tokens, float *out_logits);

/*
 * Same as tiles_decode, but prompt, out_tokens and out_logits are HOST
 * buffers (no counterpart on the pages: the end-to-end measurement): the call copies the prompt in, decodes, copies the results out and
 * synchronises `stream` before returning (so it also reports kernel errors).
 * out_logits may be NULL. Uses the plan's own device staging buffers.
 */
tiles_status_t tiles_decode_host(tiles_plan_t plan, void *k_cache, void *v_cache,
                                 const int32_t *prompt_host, int32_t n_prompt, int32_t start_pos,
                                 int32_t n_new, void *stream, int32_t *out_tokens_host,
                                 float *out_logits_host);

/*
 * tiles_decode without any device allocation. The pages have no counterpart:
 * this exists for callers that may not allocate GPU memory when they decode
 * (a process whose device memory is all handed to its own allocator, or a
 * runtime that forbids allocation after start-up), so the kernel's per-call
 * working memory comes from one fixed array compiled into the library instead
 * of the plan's own buffers. Same arguments, ownership, results and errors as
 * tiles_decode; device-side errors still go to the plan's status word
 * (read with tiles_status).
 *
 *   - The array is 1 MiB of device memory, held by every GPU that loads the
 *     library until the process exits. A plan whose working memory does not
 *     fit (q/k/v, split partials, attention output, residual, FFN activation,
 *     argmax keys and counters) is rejected with TILES_ERR_CAPACITY.
 *   - The first call on a device looks up the array's device address once
 *     and keeps it for the life of the process: make that first call before
 *     any stream capture, and make every call in the device's primary context
 *     (the runtime's default; after cudaDeviceReset or under another current
 *     context the kept address would not point at the array).
 *   - Every call on a device shares the one array and finds it as the previous
 *     call left it; the call clears what must start at zero. Calls whose work
 *     overlaps on the GPU (other streams, other plans) race on it: keep them
 *     ordered.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
tiles_status_t tiles_decode_noalloc(tiles_plan_t plan, void *k_cache, void *v_cache,
                                    const int32_t *prompt, int32_t n_prompt, int32_t start_pos,
                                    int32_t n_new, void *stream, int32_t *out_tokens,
                                    float *out_logits);

/* Synchronises `stream` and reads the plan's device status word, then clears
 * it ("Tiles", "What the code contains": the runtime's checks; kernel-side
 * waits are bounded and report here). Returns TILES_OK, TILES_ERR_TIMEOUT, TILES_ERR_DEVICE_BOUNDS or CUDA. */
tiles_status_t tiles_status(tiles_plan_t plan, void *stream);

/* Static string naming a status code (no counterpart on the pages). Never NULL. */
const char *tiles_status_string(tiles_status_t status);

/* Diagnostics (no counterpart on the pages): makes later tiles_decode calls on this plan record a per-task
 * timeline of their first `steps` steps into `trace` (device memory, caller
 * owned, at least n_ctas * steps * max_tasks_per_cta * 16 uint64 words, see
 * tiles_plan_info.max_tasks_per_cta). Word layout per task record:
 *    0 consumer wait start        1 inputs ready (after the counter wait)
 *    2 task end                   3 producer: first chunk of the task
 *    4 producer: last chunk       5 producer ns stalled on a full ring
 *    6 op | layer << 8 | chunks << 32
 *    7 prologue end (input vector gathered and normalised; attention: the
 *      first head's q/k/v ready)
 *    8 first chunk in shared memory
 *    9 attention: split partials written   10 attention: merge inputs in
 *   11..15 zero
 * Times are %globaltimer nanoseconds; a word a task does not use stays 0.
 * trace == NULL or steps == 0 turns it off. Errors: INVALID_ARG. */
tiles_status_t tiles_plan_set_trace(tiles_plan_t plan, void *trace, int32_t steps);

/* Facts about a built plan (or a host-only schedule), for reports and tests
 * (no counterpart on the pages). */
typedef struct {
    int32_t n_ctas, threads_per_cta, smem_bytes, slot_bytes, ring_slots, kv_splits;
    int32_t scheduler, n_tasks, n_counters, phases_per_step, max_tasks_per_cta;
    int32_t kv_block;           /* positions per KV chunk (a multiple of 16)                 */
    int32_t attn_tensor_cores;  /* 1: splits of >= 8 chunks give each chunk to one warp (the
                                   kernel instance carries that form); 0: every split
                                   shares its chunks across the warps. Either way every
                                   chunk is a swizzled TMA tile reduced by m16n8k16 MMAs     */
    int32_t rows_per_chunk[5];  /* GEMV rows per ring chunk: Q/K/V, O, gate/up (pairs),
                                   down, LM head                                             */
    int32_t weight_format;      /* TILES_WEIGHTS_BF16 or TILES_WEIGHTS_INT8                   */
    int32_t kv_format;          /* TILES_KV_BF16 or TILES_KV_INT8                             */
    int64_t weight_bytes_per_token;     /* every weight byte the kernel streams per step */
    int64_t max_cta_bytes, min_cta_bytes; /* per-step streamed weight bytes, busiest/idlest CTA */
} tiles_plan_info;

tiles_status_t tiles_plan_get_info(tiles_plan_t plan, tiles_plan_info *info);

/* ------------------------------------------------------------------------ */
/* Multi-token passes: verify steps and batched prompt prefill.              */

/* Tokens a single pass of tiles_forward handles; longer inputs run in
 * consecutive passes, and a verify step takes at most this many inputs. */
#define TILES_MAX_FORWARD_TOKENS 256

/*
 * Runs n_tokens input tokens through the model at positions start_pos ..
 * start_pos + n_tokens - 1 ("Tiles", "Scope and code release": batched
 * prefill instead of one token per step; "History and roadmap", "M8 so far":
 * multi-token verify steps), asynchronous on `stream`. The result is what
 * n_tokens decode steps with those inputs compute: token i attends to every
 * cached position up to its own (the K/V rows of the earlier tokens of the
 * call included), and its K/V rows are written into the caches. Each pass of
 * up to TILES_MAX_FORWARD_TOKENS tokens runs every layer for all of its
 * tokens at once: the projections as BF16 tensor-core GEMMs with FP32
 * accumulation, attention as a causal split-KV multi-query kernel, the same
 * BF16 rounding points as tiles_decode.
 *
 *   k_cache, v_cache  device, as for tiles_decode; positions < start_pos filled
 *   tokens            device, n_tokens ids in [0, vocab)
 *   out_argmax        device, n_tokens int32: the greedy token after each input
 *   out_logits        device, [n_tokens][vocab] float32, or NULL
 *
 * BF16 plans only (TILES_ERR_UNSUPPORTED for INT8 weights or an INT8 KV cache). The first call
 * allocates the plan's working memory for these passes. An out-of-range
 * token id is recorded in the status word (tiles_status). Errors:
 * INVALID_ARG, CAPACITY (start_pos + n_tokens > max_pos), UNSUPPORTED,
 * DEVICE_MISMATCH, CUDA.
 */
tiles_status_t tiles_forward(tiles_plan_t plan, void *k_cache, void *v_cache, const int32_t *tokens,
                             int32_t n_tokens, int32_t start_pos, void *stream, int32_t *out_argmax,
                             float *out_logits);

/*
 * One verify step of greedy speculative decoding ("History and roadmap",
 * "M8 so far": verify steps on the split-KV decode kernels; draft tokens
 * handed to the verify step on the device). inputs = the last emitted token
 * followed by k draft tokens d_1 .. d_k (device, k + 1 ids, k + 1 <=
 * TILES_MAX_FORWARD_TOKENS), placed at positions start_pos .. start_pos + k.
 * With a_i the greedy token after input i, the step accepts the longest
 * prefix with d_{i+1} == a_i (n drafts) and writes d_1 .. d_n, a_n to
 * out_tokens (device, k + 1 int32; n + 1 of them written) and n to
 * *out_n_accepted (device). Greedy decoding from the same state emits the
 * same tokens. K/V rows are written for all k + 1 inputs; rows after
 * start_pos + n are stale and are overwritten by the next step, which starts
 * at start_pos + n + 1 with a_n as its last token. out_logits: device
 * [k + 1][vocab] float32, or NULL. Errors as tiles_forward.
 */
tiles_status_t tiles_verify(tiles_plan_t plan, void *k_cache, void *v_cache, const int32_t *inputs, int32_t k,
                            int32_t start_pos, void *stream, int32_t *out_tokens, int32_t *out_n_accepted,
                            float *out_logits);

/* ------------------------------------------------------------------------ */
/* Schedule inspection without a GPU (planner and validator tests).          */

enum {
    TILES_OP_QKV = 1,      /* RMSNorm prologue, rows of [Wq; Wk; Wv] -> FP32 q,k,v        */
    TILES_OP_ATTN = 2,     /* q/k norm + RoPE + KV write, split-KV partial, then the merge of
                              1/S of the kv head's outputs (item = kv head * splits + split) */
    TILES_OP_COMBINE = 3,  /* unused: the attention tiles merge the splits themselves     */
    TILES_OP_OPROJ = 4,    /* rows of Wo, residual add                                    */
    TILES_OP_GATEUP = 5,   /* RMSNorm prologue, rows of Wg and Wu, SwiGLU epilogue        */
    TILES_OP_DOWN = 6,     /* rows of Wd, residual add                                    */
    TILES_OP_LMHEAD = 7,   /* final RMSNorm, rows of the tied embedding, argmax           */
    TILES_OP_SYNC = 8      /* no work: barrier arrival only (wave scheduler)              */
};

#define TILES_NO_COUNTER 0xFFFFu

/* One scheduled tile task. A CTA runs its task list once per step. Before a
 * task, the CTA waits until counter `wait_ctr` reaches
 * wait_mul * step + wait_add (step counted from the launch's first step);
 * after it, the CTA adds 1 to `signal_ctr`. */
typedef struct {
    uint8_t op;
    uint8_t phase_kind;      /* position of the op within its layer (0..5), 6 = LM head */
    uint16_t layer;
    uint32_t begin, end;     /* output rows or items                                     */
    uint16_t wait_ctr, signal_ctr;
    uint32_t wait_mul, wait_add;
} tiles_task;

typedef struct tiles_schedule_s *tiles_schedule_t;

/* Builds (but does not validate) the schedule the planner would make for
 * n_ctas CTAs, a ring of ring_slots slots of slot_bytes bytes. Host only
 * ("Tiles", intro: the offline planner's assignment and order). */
tiles_status_t tiles_schedule_build(const tiles_model_desc *desc, const tiles_plan_opts *opts,
                                    int32_t n_ctas, tiles_schedule_t *out);

/* Validates a schedule ("Tiles", "What the code contains": the planner and the
 * runtime validate the schedule): every output row / item covered exactly once per step,
 * indices in range, each wait satisfiable by earlier signals and covering all
 * of them, copy sizes and ring slots 16-byte aligned. Returns TILES_OK or
 * TILES_ERR_PLAN_INVALID; `why` (may be NULL) receives a message. */
tiles_status_t tiles_schedule_validate(tiles_schedule_t sched, char *why, size_t why_len);

/* Mutable view of the task table (fault injection in tests; no counterpart on
 * the pages): tasks of CTA c are tasks[offsets[c] .. offsets[c+1]). Valid
 * until the schedule is destroyed. */
tiles_status_t tiles_schedule_tasks(tiles_schedule_t sched, tiles_task **tasks,
                                    int32_t *n_tasks, const int32_t **offsets, int32_t *n_ctas);

/* Per-CTA weight+KV bytes streamed in one step at context position `pos`
 * ("Tiles", intro: the planner balances the bytes each worker streams). */
tiles_status_t tiles_schedule_cta_bytes(tiles_schedule_t sched, int32_t pos, int64_t *bytes);

/* The facts tiles_plan_get_info reports, for a schedule built on the host
 * (no GPU involved). Errors: INVALID_ARG on a null argument. */
tiles_status_t tiles_schedule_get_info(tiles_schedule_t sched, tiles_plan_info *info);

/* Frees a schedule (no counterpart on the pages). NULL is allowed. */
void tiles_schedule_destroy(tiles_schedule_t sched);

/* Weight-only INT8 quantization of a row-major [rows][cols] BF16 matrix (device
 * pointers), one output row per CTA, asynchronous on stream: scales[r] =
 * max_j |w_rj| / 127 and codes[r][j] = w_rj / scales[r] rounded to nearest
 * even and clamped to [-127, 127], in FP32 (an all-zero row gets scale 0 and
 * codes 0). The same kernel quantizes a plan's weights when weight_format is
 * TILES_WEIGHTS_INT8 (the plan keeps each code as the byte q + 128, which its
 * GEMV converts without a sign flip). codes: rows * cols int8; scales: rows floats; both
 * caller-owned. TILES_ERR_INVALID_ARG on a null pointer (rows > 0), rows < 0
 * or cols < 1; TILES_ERR_CUDA if the launch fails. */
tiles_status_t tiles_quantize_rows_int8(const void *w_bf16, int32_t rows, int32_t cols, void *codes,
                                        float *scales, void *stream);

/* The two caller-owned device buffers of a TILES_KV_INT8 cache ("History and
 * roadmap", "M8 so far": INT8 KV cache with smoothed keys; see TILES_KV_INT8
 * for the quantities). With Z = n_layers * n_kv_heads, d =
 * head_dim and MP = max_pos rounded up to a multiple of 16 (position strides
 * stay multiples of 16 bytes, as the kernel's tiled copies need):
 *   k buffer: key codes   int8  [Z][MP][d]  at offset 0
 *             key scales  float [Z][MP]     at k_scale_off
 *             key shifts  float [Z][d]      at k_mu_off (mu, per channel)
 *   v buffer: value codes int8  [Z][d][MP]  at offset 0 (transposed: a
 *                                          head's channel is one row)
 *             value scales float [Z][MP]    at v_scale_off
 * Offsets are multiples of 256 bytes; the buffers must be 16-byte aligned.
 * Positions max_pos..MP-1 are never read as data. Fills *out from desc
 * alone. Errors: INVALID_ARG (null argument, non-positive dimension). */
typedef struct {
    int64_t k_bytes, v_bytes;                 /* sizes of the two buffers          */
    int64_t k_scale_off, k_mu_off, v_scale_off;
    int32_t pos_stride;                       /* MP                                */
} tiles_kv8_layout;

tiles_status_t tiles_kv8_get_layout(const tiles_model_desc *desc, tiles_kv8_layout *out);

/* Builds the INT8 cache of the prefilled positions 0..n_pos-1 from BF16 caches
 * ([L][n_kv][max_pos][d], device), asynchronous on `stream` ("History and
 * roadmap", "M8 so far": smoothed keys; the plainest scheme, the pages give none): per (layer, KV
 * head) the key shift mu_j = (sum over t < n_pos of K[t][j]) / n_pos, summed
 * in FP64 in position order and rounded to FP32 (0 when n_pos = 0), then
 * every row of positions < n_pos quantized as TILES_KV_INT8 states. Other
 * positions of k8 / v8 are left as they are. Errors: INVALID_ARG (null
 * pointer, n_pos outside [0, max_pos], unaligned buffer), UNSUPPORTED
 * (head_dim not 64 or 128), CUDA. */
tiles_status_t tiles_kv8_from_bf16(const tiles_model_desc *desc, const void *k_bf16, const void *v_bf16,
                                   int32_t n_pos, void *k8, void *v8, void *stream);

/* ------------------------------------------------------------------------ */
/* Measurement helpers.                                                       */

/* Device-to-device copy of `bytes` (multiple of 16, both pointers 16-byte
 * aligned) by a grid of n_ctas CTAs (0 = 2 per SM), asynchronous on stream.
 * The HBM peak the roofline fraction is taken against ("History and roadmap",
 * "Where it stands": kernels measured against their memory roofline). */
tiles_status_t tiles_copy_bw(void *dst, const void *src, size_t bytes, int32_t n_ctas,
                             void *stream);

/* Grid-barrier round trip ("Tiles", intro: the cost of a barrier between
 * waves): one cooperative launch of n_ctas CTAs that crosses
 * `rounds` grid barriers; *ns_per_barrier receives the mean cost measured
 * inside the kernel with the global timer. Synchronous. */
tiles_status_t tiles_barrier_cost(int32_t n_ctas, int32_t rounds, double *ns_per_barrier);

#ifdef __cplusplus
}
#endif
#endif /* TILES_H */

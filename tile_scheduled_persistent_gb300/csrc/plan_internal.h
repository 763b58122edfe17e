// The plan object behind tiles_plan_t (host side), shared by the decode
// runtime and the multi-token forward pass.
#pragma once

#include <vector>

#include "tiles_internal.h"

// Working memory of the multi-token forward pass (tiles_forward,
// tiles_verify), allocated on first use for up to TILES_MAX_FORWARD_TOKENS tokens
// per pass.
struct ForwardScratch {
    std::vector<void *> allocs;
    bool ready = false;
    uint16_t *x = nullptr;        // residual stream [T][H] bf16
    uint16_t *h = nullptr;        // normed GEMM input [T][H] bf16
    uint16_t *q = nullptr;        // roped queries [T][nq d] bf16
    uint16_t *o = nullptr;        // attention output [T][nq d] bf16
    uint16_t *a = nullptr;        // SwiGLU output [T][F] bf16
    float *part = nullptr;        // GEMM split-K partial sums
    size_t part_elems = 0;
    float *apart = nullptr;       // attention split partials [T nq][splits][2 + d]
    size_t attn_pairs = 0;        // (token, split) pairs apart holds
    float *logits = nullptr;      // [T][V] when the caller passes none
    int32_t *argmax = nullptr;    // [T]
    int32_t *tokens = nullptr;    // staging of verify inputs
};

struct tiles_plan_s {
    tiles_schedule_s sched;
    int device = -1, sm_count = 0, cc_major = 0, cc_minor = 0;
    std::vector<void *> allocs;
    tiles::KernelParams base{};
    unsigned long long *d_keys = nullptr;  // keys then counters: one memset per launch
    size_t sync_bytes = 0;
    int32_t *d_prompt_stage = nullptr, *d_tokens_stage = nullptr;
    float *d_logits_stage = nullptr;
    size_t logits_stage_elems = 0;
    std::vector<tiles::LayerPtrs> layers_host;  // the device table's pointers, for host launches
    ForwardScratch fwd;
};

// TILES_OK when the current device is the plan's (same device, same SM count).
extern "C" tiles_status_t plan_check_device(tiles_plan_t plan);

// The plan object behind tiles_plan_t (host side), shared by the decode
// runtime and the multi-token forward pass.
#pragma once

#include <stddef.h>

#include <array>
#include <utility>
#include <vector>

#include "tiles_internal.h"

#ifdef __CUDACC__
#include <cuda_runtime.h>
namespace tiles {
namespace fwd {
// Tensor-core projections of the multi-token pass (gemm_tc.cu): tiles of
// kTcM weight rows against all T tokens (n_tile = T rounded up to 16), K
// split into sk ranges of kps elements, `stages` shared-memory stages.
constexpr int kTcM = 128;
struct TcShape {
    int n_tile, mt, sk, kps, stages;
    size_t smem;
};
TcShape tc_shape(int M, int T, int K, int sms, int max_sk);
cudaError_t gemm_tc_configure();
// act: null, or (one split only, M even, rows in gate/up pairs) the SwiGLU
// output bf16 [T][M / 2] in place of C
cudaError_t gemm_tc_launch(const TensorMap &mw, const TensorMap &mx, const TcShape &s, int M, int T, int K,
                           float *C, uint16_t *act, uint32_t *status, unsigned long long timeout_ns,
                           cudaStream_t st);
}  // namespace fwd
}  // namespace tiles
#endif

namespace tiles {
// A 2-D BF16 tensor map (runtime.cu): `rows` rows of `inner` elements,
// `row_bytes` apart, boxes of box_inner x box_rows elements, 128-byte swizzle,
// rows past the end read as zeros. False if the driver refuses it.
bool encode_bf16_2d(TensorMap *out, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_rows);
}  // namespace tiles

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
    unsigned long long *arg_keys = nullptr;  // [T] running argmax keys (zero between passes)
    uint32_t *arg_tickets = nullptr;         // [T] blocks done per token (zero between passes)
    // tensor maps of the projections' operands: (base, inner, rows, row bytes, box rows) -> map
    std::vector<std::pair<std::array<uint64_t, 5>, tiles::TensorMap>> maps;
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

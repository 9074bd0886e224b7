// draft_tc.cuh -- the tensor-core (tcgen05) Markov-head kernels: interface.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

struct DraftTcArgs {
    const void* U;
    // fused drafter logits (d > 0): hidden states h [R, gamma, d] and the shared
    // lm_head W_lm [V, d] (bf16) in place of U
    const void* h = nullptr;
    const void* W_lm = nullptr;
    int d = 0;
    const void* W1;
    const void* W2;
    const int32_t* anchor;
    const uint64_t* seeds;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank;
    int32_t* y;
    float* q_lse;
    float* q_tok;
    float* q_logits;
    int32_t* dev_status;
    void* ws;
};

// The extra token of every request after the verify decisions, with the
// drafter's logits of the rejected row recomputed from its Markov factors.
// The per-request rows (residual_tc_rows of the workspace) are written by the
// verify decisions and the keys (residual_tc_keys) zeroed by its prologue.
struct ResidualTcArgs {
    const void* U;
    const void* W1;
    const void* W2;
    const uint64_t* seeds;
    uint32_t cycle;
    float invT;
    int R, gamma, V, rank;
    const float* target;       // packed target rows
    int32_t* out_tokens;       // [R, gamma + 1]
    int32_t* dev_status;
    void* ws;
};

bool draft_tc_supported(int u_dtype, int w_dtype, int R, int V, int rank);
// the draft's one cooperative launch needs a CTA per SM for every 128 requests
bool draft_tc_fits(int R);
size_t draft_tc_workspace(int R, int gamma, int rank);
int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream);

size_t residual_tc_workspace(int R, int rank);
// the per-request rows and winner keys inside the residual workspace (both
// prepared by the verify kernels: rows as requests are decided, keys zeroed)
ResRow* residual_tc_rows(void* ws, int R);
unsigned long long* residual_tc_keys(void* ws, int R);
int launch_residual_tc(const ResidualTcArgs& a, cudaStream_t stream);

}  // namespace dspark

// draft_tc.cuh -- the tensor-core (tcgen05) Markov draft: interface.
#pragma once

#include "common.cuh"

namespace dspark {

struct DraftTcArgs {
    const void* U;
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

bool draft_tc_supported(int u_dtype, int w_dtype, int R, int V, int rank);
size_t draft_tc_workspace(int R, int V, int rank);
int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream);

}  // namespace dspark

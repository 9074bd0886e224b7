// kernels.cuh -- launch parameters and entry points of the library's kernels.
#pragma once

#include "common.cuh"

namespace dspark {

// ----------------------------------------------------------------------------
// Verify
// ----------------------------------------------------------------------------
constexpr int kVerifyThreads = 256;
constexpr int kVerifyChunk = 8192;  // target-row elements per CTA unit of the extra-token draw
constexpr int kStatChunk = 1024;    // target-row elements per warp unit of the row statistics

struct RowStat {  // per (row, chunk): max and sum of exp(t - max), first argmax
    float m, s;
    int idx, pad;
};
struct VerifyJob {  // per request: the row the extra token comes from
    int row, pos, mode, pad;  // mode 0: none, 1: residual, 2: bonus
    float lse;
    float pad2[3];
};
struct SamplePartial {  // per (request, chunk) of a Gumbel-max draw
    float best;
    int idx;
    float best_alt;  // noise on p instead of the residual (empty-residual fallback)
    int idx_alt;
    float mass;      // residual mass seen
    float pad[3];
};

// Per request after the verify decisions, for the residual draw of
// dspark_verify_markov: what it draws and the A row of its recomputed logits.
struct ResRow {
    int mode;      // 0: nothing to draw, 1: residual of row pos, 2: bonus from p of row pos
    int pos;       // block position of the row
    int trow;      // packed target row
    uint32_t w3;   // Philox counter word 3 (cycle and purpose)
    float lse2_p;  // target log-normaliser of the row (scaled logits), base 2
    float q_lse2;  // drafter log-normaliser at pos (mode 1), base 2
    int prev;      // token whose W1 row is the A row (mode 1), else -1
    float pad;
};

struct VerifyParams {
    const float* target;
    const int32_t* cu;
    const int32_t* y;
    const float* q_logits;
    const float* q_lse;
    const float* q_tok;
    const uint64_t* seeds;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, max_rows, nchunk, nsub;
    int32_t* n_acc;
    int32_t* out_tokens;
    float* p_tok;
    int32_t* dev_status;
    // workspace
    int* ok;        // [1] cu_seqlens well formed
    int* valid;     // [R]
    int* cnt1;      // [R]
    int* cnt2;      // [R]
    int* act;       // [2][R] requests still drafting-accepted, per round parity
    int* lazy;      // [8] round state of the verify pass: barrier count and generation,
                    // next-round counts (2), abort flag
    RowStat* stats; // [2][R * nsub] per (round parity, request, kStatChunk-element unit of its row)
    VerifyJob* jobs;        // [R]
    SamplePartial* parts;   // [R * nchunk]
    // dspark_verify_markov only (else NULL): the residual rows, written as the
    // requests are decided, and what they need
    ResRow* res_rows = nullptr;       // [R]
    unsigned long long* res_keys = nullptr;  // [R + 1] the residual draw's winner keys and its count of
                                             // CTAs done, zeroed by the prologue
    const int32_t* anchor = nullptr;  // [R]
    const uint16_t* W1 = nullptr;     // [V, rank] bf16: each predecessor's row is requested into L2
    int rank = 0;
    // target rows in pinned host memory (dspark_verify_markov): every row the
    // decision pass streams is also stored here, [R, V], so that the residual
    // launch reads each request's last row from device memory
    float* row_copy = nullptr;
    // the grid barriers between rounds: wait limit, and an arrival count one
    // above the grid's when the barrier-timeout test injection is on
    unsigned long long wait_ns = 2000000000ull;
    int phantom = 0;
};

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream);
// prologue + stats/decision passes only (the extra token is left to the caller)
cudaError_t launch_verify_decide(const VerifyParams& p, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Draft (CUDA-core path)
// ----------------------------------------------------------------------------
constexpr int kDraftThreads = 256;
constexpr int kDraftChunk = 8192;

struct DraftPartial {
    float score;
    int idx;
    float s_at;  // the logit s of the chosen index
    float m, sum;
    float pad[3];
};

struct DraftParams {
    const void* U;
    int u_dtype;
    const void* W1;
    const void* W2;
    int w_dtype;
    const int32_t* anchor;
    const uint64_t* seeds;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank, nchunk;
    int32_t* y;
    float* q_lse;
    float* q_tok;
    float* q_logits;
    int32_t* dev_status;
    // workspace
    int* cnt;            // [R]
    DraftPartial* parts; // [R * nchunk]
    float* bias;         // [R * V]
};

cudaError_t launch_draft_simt(const DraftParams& p, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Selection and commit
// ----------------------------------------------------------------------------
constexpr int kSelectThreads = 1024;
constexpr int kSelectMaxItems = 8192;
constexpr int kSelectMaxSteps = 64;

struct SelectParams {
    const float* c;              // plan: c_seq [n_cycles, R, gamma]
    const float* c_hist;
    const int32_t* capture_sizes;
    const float* sps;
    int n_steps, K_cap, mode, R, gamma;
    float conf_min;              // the cutoff modes' threshold
    float* a;
    int32_t* l;                  // plan: [n_cycles, R]
    int32_t* cu;
    int32_t* K_used;             // plan: [n_cycles]
    int32_t* dev_status;
    // plan only
    int lag = 0;
    const int32_t* n_full = nullptr;  // [n_cycles, R] or NULL
    double* stats = nullptr;          // [n_cycles, 4]
};

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);
cudaError_t launch_plan(const SelectParams& p, int n_cycles, cudaStream_t stream);

cudaError_t launch_philox_batch(const uint32_t* ctr, const uint64_t* keys, int n, uint32_t* out,
                                cudaStream_t stream);

// Process-wide settings of the grid-wide waits (dspark_set_wait_limit_ns,
// dspark_set_fault_injection), read by each call when it is enqueued.
unsigned long long grid_wait_limit_ns();
unsigned fault_injection_mask();

// ----------------------------------------------------------------------------
// Confidence calibration (sequential temperature scaling)
// ----------------------------------------------------------------------------
constexpr int kCalMaxCtas = 64;  // CTAs per position
size_t calibrate_workspace(int gamma);
cudaError_t launch_calibrate(const float* z, const uint8_t* accepted, int N, int gamma, float* tau, double* nll,
                             int32_t* count, int32_t* dev_status, void* ws, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Paged KV bookkeeping around a verify
// ----------------------------------------------------------------------------
cudaError_t launch_kv_reserve(const int32_t* kv_len, const int32_t* l, int R, int P, int32_t* bt, int max_blocks,
                              const int32_t* free_pages, int32_t* free_top, int pool_pages, int32_t* reserved,
                              int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_kv_commit(int32_t* kv_len, const int32_t* l, const int32_t* n_acc, int R, int P, int32_t* bt,
                             int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages,
                             int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_commit(const int32_t* n_acc, const int32_t* l, int R, int gamma,
                          int32_t* commit_len, int32_t* cu_commit, int32_t* discard,
                          int32_t* total, int32_t* dev_status, cudaStream_t stream);

}  // namespace dspark

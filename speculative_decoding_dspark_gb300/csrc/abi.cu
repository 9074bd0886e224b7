// abi.cu -- the library's extern "C" entry points (declared in dspark.h).
//
// Host-side argument checks, workspace carving and kernel dispatch only; every
// step of the cycle runs in the kernels.  No call allocates memory,
// synchronises or throws; the only state is the pair of process-wide wait
// settings (limit of the grid-wide waits, test injection), read at each call.
#include <atomic>
#include <cstring>

#include "kernels.cuh"
#include "draft_tc.cuh"

namespace {

using namespace dspark;

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

// ---- workspace layouts (the size query and the calls share them) ------------
struct DraftSimtLayout {
    size_t cnt, parts, bias, total;
};
DraftSimtLayout draft_simt_layout(int R, int V) {
    DraftSimtLayout L;
    const int nchunk = (V + kDraftChunk - 1) / kDraftChunk;
    size_t off = 0;
    L.cnt = off; off += align_up(sizeof(int) * (size_t)R);
    L.parts = off; off += align_up(sizeof(DraftPartial) * (size_t)R * nchunk);
    L.bias = off; off += align_up(sizeof(float) * (size_t)R * V);
    L.total = off;
    return L;
}

struct VerifyLayout {
    size_t ok, valid, cnt1, cnt2, act, lazy, stats, jobs, parts, total;
};
// (The rows are streamed lazily, so the scratch does not grow with max_rows.)
VerifyLayout verify_layout(int R, int V) {
    VerifyLayout L;
    const int nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
    size_t off = 0;
    L.ok = off; off += align_up(sizeof(int));
    L.valid = off; off += align_up(sizeof(int) * (size_t)R);
    L.cnt1 = off; off += align_up(sizeof(int) * (size_t)R);
    L.cnt2 = off; off += align_up(sizeof(int) * (size_t)R);
    L.act = off; off += align_up(sizeof(int) * 2 * (size_t)R);
    L.lazy = off; off += align_up(sizeof(int) * 8);
    const int nsub = (V + kStatChunk - 1) / kStatChunk;
    L.stats = off; off += align_up(sizeof(RowStat) * 2 * (size_t)R * nsub);  // two rounds in flight
    L.jobs = off; off += align_up(sizeof(VerifyJob) * (size_t)R);
    L.parts = off; off += align_up(sizeof(SamplePartial) * (size_t)R * nchunk);
    L.total = off;
    return L;
}

template <typename T>
T* carve(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<unsigned char*>(ws) + off);
}

bool tc_applies(int u_dtype, int w_dtype, int R, int V, int rank, unsigned flags) {
    if (flags & DSPARK_DRAFT_FORCE_SIMT) return false;
    return draft_tc_supported(u_dtype, w_dtype, R, V, rank) && draft_tc_fits(R);
}

bool valid_dtype(int d) { return d == DSPARK_F32 || d == DSPARK_BF16; }

// Where a caller's pointer lives: device (or managed) memory, pinned host memory
// the device can read, or memory the device cannot be trusted to read.
enum class Residence { kDevice, kPinnedHost, kOther };
Residence residence(const void* ptr) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of the query
        return Residence::kOther;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return Residence::kDevice;
    if (at.type == cudaMemoryTypeHost && at.devicePointer == ptr) return Residence::kPinnedHost;
    return Residence::kOther;
}

// Process-wide settings of the grid-wide waits (see dspark_set_wait_limit_ns).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<unsigned> g_inject{0u};

}  // namespace

namespace dspark {
unsigned long long grid_wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
unsigned fault_injection_mask() { return g_inject.load(std::memory_order_relaxed); }
}  // namespace dspark

extern "C" {

uint64_t dspark_set_wait_limit_ns(uint64_t limit_ns) {
    if (limit_ns == 0 || limit_ns > kDefaultWaitNs) limit_ns = kDefaultWaitNs;
    return g_wait_ns.exchange(limit_ns);
}

unsigned dspark_set_fault_injection(unsigned mask) {
    return g_inject.exchange(mask & (DSPARK_INJECT_VERIFY_BARRIER | DSPARK_INJECT_DRAFT_BARRIER));
}

const char* dspark_status_string(int status) {
    switch (status) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case DSPARK_ERR_CAPACITY: return "capacity exceeded";
        case DSPARK_ERR_CUDA: return "CUDA error";
        case DSPARK_ERR_TIMEOUT: return "device wait timed out";
        case DSPARK_ERR_DEVICE_INPUT: return "bad device-side input (token id, length or confidence)";
        case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DSPARK_ERR_BOUNDS: return "device-side bounds check failed (debug build)";
        default: return "unknown status";
    }
}

int dspark_version(void) { return 10200; }

int dspark_markov_draft_uses_tensor_cores(int u_dtype, int w_dtype, int R, int V, int rank,
                                          unsigned flags) {
    return tc_applies(u_dtype, w_dtype, R, V, rank, flags) ? 1 : 0;
}

size_t dspark_workspace_size(int op, int R, int gamma, int V, int rank, int max_rows,
                             int w_dtype, unsigned flags) {
    if (op == DSPARK_OP_CALIBRATE) return (gamma <= 0 || gamma > 16) ? 0 : calibrate_workspace(gamma);
    if (R <= 0) return 0;
    switch (op) {
        case DSPARK_OP_DRAFT:
            if (V <= 0 || rank <= 0 || gamma <= 0) return 0;
            if (tc_applies(w_dtype, w_dtype, R, V, rank, flags)) return draft_tc_workspace(R, gamma, rank);
            return draft_simt_layout(R, V).total;
        case DSPARK_OP_VERIFY:
            if (V <= 0 || max_rows < 0) return 0;
            return verify_layout(R, V).total;
        case DSPARK_OP_VERIFY_MARKOV: {
            if (V <= 0 || max_rows < 0 || rank <= 0) return 0;
            const size_t base = align_up(verify_layout(R, V).total) + residual_tc_workspace(R, rank);
            // a host-resident target keeps each request's latest row on the device
            return (flags & DSPARK_VERIFY_HOST_TARGET) ? align_up(base) + align_up(sizeof(float) * (size_t)R * V) : base;
        }
        case DSPARK_OP_DRAFT_FUSED:
            if (V <= 0 || rank <= 0 || gamma <= 0) return 0;
            return draft_tc_workspace(R, gamma, rank);
        case DSPARK_OP_SELECT:
            return 0;
        default:
            return 0;
    }
}

int dspark_markov_draft(const void* U, int u_dtype, const void* W1, const void* W2,
                        int w_dtype, const int32_t* anchor, const uint64_t* seeds,
                        uint32_t cycle, float temperature, int R, int gamma, int V,
                        int rank, int32_t* draft_tokens, float* q_lse, float* q_tok,
                        float* q_logits, unsigned flags, void* ws, size_t ws_bytes,
                        int32_t* dev_status, dspark_stream_t stream) {
    if (!U || !W1 || !W2 || !anchor || !draft_tokens) return DSPARK_ERR_INVALID_ARG;
    if (!valid_dtype(u_dtype) || !valid_dtype(w_dtype)) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || V <= 0 || rank <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARG;
    if (cycle >= (1u << 28)) return DSPARK_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!seeds || !q_lse || !q_tok)) return DSPARK_ERR_INVALID_ARG;
    if ((flags & ~DSPARK_DRAFT_FORCE_SIMT) != 0) return DSPARK_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DSPARK_ERR_WORKSPACE;
    const float invT = greedy ? 1.0f : 1.0f / temperature;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (tc_applies(u_dtype, w_dtype, R, V, rank, flags)) {
        if (ws_bytes < draft_tc_workspace(R, gamma, rank)) return DSPARK_ERR_WORKSPACE;
        if (!aligned16(U) || !aligned16(W1) || !aligned16(W2)) return DSPARK_ERR_UNSUPPORTED;
        DraftTcArgs a;
        a.U = U; a.W1 = W1; a.W2 = W2; a.anchor = anchor; a.seeds = seeds; a.cycle = cycle;
        a.invT = invT; a.greedy = greedy; a.R = R; a.gamma = gamma; a.V = V; a.rank = rank;
        a.y = draft_tokens; a.q_lse = q_lse; a.q_tok = q_tok; a.q_logits = q_logits;
        a.dev_status = dev_status; a.ws = ws;
        return launch_draft_tc(a, s);
    }

    const DraftSimtLayout L = draft_simt_layout(R, V);
    if (ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    DraftParams p;
    p.U = U; p.u_dtype = u_dtype; p.W1 = W1; p.W2 = W2; p.w_dtype = w_dtype;
    p.anchor = anchor; p.seeds = seeds; p.cycle = cycle; p.invT = invT; p.greedy = greedy;
    p.R = R; p.gamma = gamma; p.V = V; p.rank = rank;
    p.nchunk = (V + kDraftChunk - 1) / kDraftChunk;
    p.y = draft_tokens; p.q_lse = q_lse; p.q_tok = q_tok; p.q_logits = q_logits;
    p.dev_status = dev_status;
    p.cnt = carve<int>(ws, L.cnt);
    p.parts = carve<DraftPartial>(ws, L.parts);
    p.bias = carve<float>(ws, L.bias);
    return cuda_status(launch_draft_simt(p, s));
}

int dspark_markov_draft_fused(const void* h, const void* W_lm, int d, const void* W1, const void* W2,
                              const int32_t* anchor, const uint64_t* seeds, uint32_t cycle,
                              float temperature, int R, int gamma, int V, int rank,
                              int32_t* draft_tokens, float* q_lse, float* q_tok, float* q_logits,
                              void* ws, size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
    if (!h || !W_lm || !W1 || !W2 || !anchor || !draft_tokens) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || V <= 0 || rank <= 0 || d <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARG;
    if (cycle >= (1u << 28)) return DSPARK_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!seeds || !q_lse || !q_tok)) return DSPARK_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DSPARK_ERR_WORKSPACE;
    // tensor cores only: the hidden size in whole 64-element k-blocks, the Markov
    // factors as for the tensor-core draft
    if (d % 64 != 0 || d > DSPARK_FUSED_MAX_D) return DSPARK_ERR_UNSUPPORTED;
    if (!draft_tc_supported(DSPARK_BF16, DSPARK_BF16, R, V, rank) || !draft_tc_fits(R)) return DSPARK_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(W_lm) || !aligned16(W1) || !aligned16(W2)) return DSPARK_ERR_UNSUPPORTED;
    if (ws_bytes < draft_tc_workspace(R, gamma, rank)) return DSPARK_ERR_WORKSPACE;
    DraftTcArgs a;
    a.U = nullptr; a.h = h; a.W_lm = W_lm; a.d = d;
    a.W1 = W1; a.W2 = W2; a.anchor = anchor; a.seeds = seeds; a.cycle = cycle;
    a.invT = greedy ? 1.0f : 1.0f / temperature; a.greedy = greedy;
    a.R = R; a.gamma = gamma; a.V = V; a.rank = rank;
    a.y = draft_tokens; a.q_lse = q_lse; a.q_tok = q_tok; a.q_logits = q_logits;
    a.dev_status = dev_status; a.ws = ws;
    return launch_draft_tc(a, reinterpret_cast<cudaStream_t>(stream));
}

int dspark_verify(const float* target_logits, const int32_t* cu_seqlens,
                  const int32_t* draft_tokens, const float* q_logits, const float* q_lse,
                  const float* q_tok, const uint64_t* seeds, uint32_t cycle,
                  float temperature, int R, int gamma, int V, int max_rows,
                  int32_t* n_accepted, int32_t* out_tokens, float* p_tok, void* ws,
                  size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
    if (!target_logits || !cu_seqlens || !draft_tokens || !n_accepted || !out_tokens)
        return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || V <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    if (R > DSPARK_VERIFY_MAX_R) return DSPARK_ERR_UNSUPPORTED;
    if (max_rows < R || (long long)max_rows > (long long)R * (gamma + 1)) return DSPARK_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARG;
    if (cycle >= (1u << 28)) return DSPARK_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!q_logits || !q_lse || !q_tok || !seeds)) return DSPARK_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DSPARK_ERR_WORKSPACE;
    const VerifyLayout L = verify_layout(R, V);
    if (ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    const int nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
    if ((long long)max_rows * ((V + kStatChunk - 1) / kStatChunk) >= (1LL << 31) ||
        (long long)R * nchunk >= (1LL << 31))
        return DSPARK_ERR_UNSUPPORTED;
    if (residence(target_logits) != Residence::kDevice) return DSPARK_ERR_UNSUPPORTED;

    VerifyParams p;
    p.target = target_logits; p.cu = cu_seqlens; p.y = draft_tokens; p.q_logits = q_logits;
    p.q_lse = q_lse; p.q_tok = q_tok; p.seeds = seeds; p.cycle = cycle;
    p.invT = greedy ? 1.0f : 1.0f / temperature; p.greedy = greedy;
    p.R = R; p.gamma = gamma; p.V = V; p.max_rows = max_rows; p.nchunk = nchunk;
    p.nsub = (V + kStatChunk - 1) / kStatChunk;
    p.n_acc = n_accepted; p.out_tokens = out_tokens; p.p_tok = p_tok; p.dev_status = dev_status;
    p.ok = carve<int>(ws, L.ok);
    p.valid = carve<int>(ws, L.valid);
    p.cnt1 = carve<int>(ws, L.cnt1);
    p.cnt2 = carve<int>(ws, L.cnt2);
    p.act = carve<int>(ws, L.act);
    p.lazy = carve<int>(ws, L.lazy);
    p.stats = carve<RowStat>(ws, L.stats);
    p.jobs = carve<VerifyJob>(ws, L.jobs);
    p.parts = carve<SamplePartial>(ws, L.parts);
    return cuda_status(launch_verify(p, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_verify_markov(const float* target_logits, const int32_t* cu_seqlens,
                         const int32_t* draft_tokens, const void* U, const void* W1,
                         const void* W2, const int32_t* anchor, int rank, const float* q_lse,
                         const float* q_tok, const uint64_t* seeds, uint32_t cycle,
                         float temperature, int R, int gamma, int V, int max_rows,
                         int32_t* n_accepted, int32_t* out_tokens, float* p_tok, void* ws,
                         size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
    if (!target_logits || !cu_seqlens || !draft_tokens || !n_accepted || !out_tokens)
        return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || V <= 0 || gamma <= 0 || gamma > 16 || rank <= 0) return DSPARK_ERR_INVALID_ARG;
    if (R > DSPARK_VERIFY_MAX_R) return DSPARK_ERR_UNSUPPORTED;
    if (max_rows < R || (long long)max_rows > (long long)R * (gamma + 1)) return DSPARK_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARG;
    if (cycle >= (1u << 28)) return DSPARK_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!U || !W1 || !W2 || !anchor || !q_lse || !q_tok || !seeds)) return DSPARK_ERR_INVALID_ARG;
    if (!draft_tc_supported(DSPARK_BF16, DSPARK_BF16, R, V, rank)) return DSPARK_ERR_UNSUPPORTED;
    if (!greedy && (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(target_logits)))
        return DSPARK_ERR_UNSUPPORTED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DSPARK_ERR_WORKSPACE;
    const Residence where = residence(target_logits);
    if (where == Residence::kOther) return DSPARK_ERR_UNSUPPORTED;
    const bool host_target = where == Residence::kPinnedHost && !greedy;
    const VerifyLayout L = verify_layout(R, V);
    const size_t res_off = align_up(L.total);
    const size_t copy_off = align_up(res_off + residual_tc_workspace(R, rank));
    if (ws_bytes < (host_target ? copy_off + sizeof(float) * (size_t)R * V : res_off + residual_tc_workspace(R, rank)))
        return DSPARK_ERR_WORKSPACE;
    const int nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
    if ((long long)max_rows * ((V + kStatChunk - 1) / kStatChunk) >= (1LL << 31)) return DSPARK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    VerifyParams p;
    p.target = target_logits; p.cu = cu_seqlens; p.y = draft_tokens; p.q_logits = nullptr;
    p.q_lse = q_lse; p.q_tok = q_tok; p.seeds = seeds; p.cycle = cycle;
    p.invT = greedy ? 1.0f : 1.0f / temperature; p.greedy = greedy;
    p.R = R; p.gamma = gamma; p.V = V; p.max_rows = max_rows; p.nchunk = nchunk;
    p.nsub = (V + kStatChunk - 1) / kStatChunk;
    p.n_acc = n_accepted; p.out_tokens = out_tokens; p.p_tok = p_tok; p.dev_status = dev_status;
    p.ok = carve<int>(ws, L.ok);
    p.valid = carve<int>(ws, L.valid);
    p.cnt1 = carve<int>(ws, L.cnt1);
    p.cnt2 = carve<int>(ws, L.cnt2);
    p.act = carve<int>(ws, L.act);
    p.lazy = carve<int>(ws, L.lazy);
    p.stats = carve<RowStat>(ws, L.stats);
    p.jobs = carve<VerifyJob>(ws, L.jobs);
    p.parts = carve<SamplePartial>(ws, L.parts);
    if (!greedy) {  // the decisions write the residual draw's per-request rows
        p.res_rows = residual_tc_rows(static_cast<unsigned char*>(ws) + res_off, R);
        p.res_keys = residual_tc_keys(static_cast<unsigned char*>(ws) + res_off, R);
        p.anchor = anchor;
        p.W1 = static_cast<const uint16_t*>(W1);
        p.rank = rank;
        if (host_target) p.row_copy = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + copy_off);
    }
    const cudaError_t e = launch_verify_decide(p, s);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    if (greedy) return DSPARK_OK;  // the decision pass already wrote the argmax token

    ResidualTcArgs a;
    a.U = U; a.W1 = W1; a.W2 = W2; a.seeds = seeds;
    a.cycle = cycle; a.invT = p.invT; a.R = R; a.gamma = gamma; a.V = V; a.rank = rank;
    a.target = host_target ? p.row_copy : target_logits;  // rows by request (host target) or packed
    a.out_tokens = out_tokens; a.dev_status = dev_status;
    a.ws = static_cast<unsigned char*>(ws) + res_off;
    return launch_residual_tc(a, s);
}

int dspark_select_prefix(const float* c, const float* c_hist, const int32_t* capture_sizes,
                         const float* sps, int n_steps, int K_cap, int mode, float conf_min, int R,
                         int gamma, float* a, int32_t* l, int32_t* cu_seqlens, int32_t* K_used,
                         void* ws, size_t ws_bytes, int32_t* dev_status,
                         dspark_stream_t stream) {
    (void)ws; (void)ws_bytes;
    if (!c || !a || !l || !cu_seqlens || !K_used) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    if (mode < DSPARK_SELECT_FIXED || mode > DSPARK_SELECT_SURVIVAL_CUTOFF) return DSPARK_ERR_INVALID_ARG;
    if (mode == DSPARK_SELECT_HISTORY && !c_hist) return DSPARK_ERR_INVALID_ARG;
    const bool planned = mode >= DSPARK_SELECT_HISTORY && mode <= DSPARK_SELECT_FIRST_STOP;
    if (planned && (n_steps <= 0 || n_steps > kSelectMaxSteps || !capture_sizes || !sps))
        return DSPARK_ERR_INVALID_ARG;
    if (mode >= DSPARK_SELECT_CONF_CUTOFF && !(conf_min == conf_min)) return DSPARK_ERR_INVALID_ARG;
    if ((long long)R * gamma > kSelectMaxItems) return DSPARK_ERR_UNSUPPORTED;
    if (K_cap < R) return DSPARK_ERR_CAPACITY;
    SelectParams p;
    p.c = c; p.c_hist = c_hist; p.capture_sizes = capture_sizes; p.sps = sps;
    p.n_steps = planned ? n_steps : 0;
    p.K_cap = K_cap; p.mode = mode; p.R = R; p.gamma = gamma; p.conf_min = conf_min;
    p.a = a; p.l = l; p.cu = cu_seqlens; p.K_used = K_used; p.dev_status = dev_status;
    return cuda_status(launch_select(p, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_plan_cycles(const float* c_seq, const int32_t* n_full, const int32_t* capture_sizes,
                       const float* sps, int n_steps, int K_cap, int mode, float conf_min, int lag,
                       int n_cycles, int R, int gamma, int32_t* l_seq, int32_t* K_seq, double* stats,
                       int32_t* dev_status, dspark_stream_t stream) {
    if (!c_seq || !capture_sizes || !sps || !l_seq || !K_seq || !stats) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || gamma > 16 || n_cycles <= 0 || lag < 1) return DSPARK_ERR_INVALID_ARG;
    if (n_cycles > (1 << 20)) return DSPARK_ERR_UNSUPPORTED;
    if (mode < DSPARK_SELECT_FIXED || mode > DSPARK_SELECT_SURVIVAL_CUTOFF) return DSPARK_ERR_INVALID_ARG;
    if (n_steps <= 0 || n_steps > kSelectMaxSteps) return DSPARK_ERR_INVALID_ARG;
    if (mode >= DSPARK_SELECT_CONF_CUTOFF && !(conf_min == conf_min)) return DSPARK_ERR_INVALID_ARG;
    if ((long long)R * gamma > kSelectMaxItems) return DSPARK_ERR_UNSUPPORTED;
    if (K_cap < R) return DSPARK_ERR_CAPACITY;
    SelectParams p;
    p.c = c_seq; p.c_hist = nullptr; p.capture_sizes = capture_sizes; p.sps = sps;
    p.n_steps = n_steps; p.K_cap = K_cap; p.mode = mode; p.R = R; p.gamma = gamma; p.conf_min = conf_min;
    p.a = nullptr; p.l = l_seq; p.cu = nullptr; p.K_used = K_seq; p.dev_status = dev_status;
    p.lag = lag; p.n_full = n_full; p.stats = stats;
    return cuda_status(launch_plan(p, n_cycles, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_fit_temperatures(const float* z, const uint8_t* accepted, int N, int gamma, float* tau,
                            double* nll, int32_t* count, void* ws, size_t ws_bytes, int32_t* dev_status,
                            dspark_stream_t stream) {
    if (!z || !accepted || !tau) return DSPARK_ERR_INVALID_ARG;
    if (N <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DSPARK_ERR_WORKSPACE;
    if (ws_bytes < calibrate_workspace(gamma)) return DSPARK_ERR_WORKSPACE;
    return cuda_status(launch_calibrate(z, accepted, N, gamma, tau, nll, count, dev_status, ws,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_kv_reserve(const int32_t* kv_len, const int32_t* l, int R, int page_size, int32_t* block_table,
                      int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages, int32_t* reserved,
                      int32_t* dev_status, dspark_stream_t stream) {
    if (!kv_len || !l || !block_table || !free_pages || !free_top) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || page_size <= 0 || max_blocks <= 0 || pool_pages < 0) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_kv_reserve(kv_len, l, R, page_size, block_table, max_blocks, free_pages, free_top,
                                         pool_pages, reserved, dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_kv_commit(int32_t* kv_len, const int32_t* l, const int32_t* n_accepted, int R, int page_size,
                     int32_t* block_table, int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages,
                     int32_t* dev_status, dspark_stream_t stream) {
    if (!kv_len || !l || !n_accepted || !block_table || !free_pages || !free_top) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || page_size <= 0 || max_blocks <= 0 || pool_pages < 0) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_kv_commit(kv_len, l, n_accepted, R, page_size, block_table, max_blocks, free_pages,
                                        free_top, pool_pages, dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_philox4x32_10(const uint32_t* ctr, const uint64_t* keys, int n, uint32_t* out,
                         dspark_stream_t stream) {
    if (n < 0 || (n > 0 && (!ctr || !keys || !out))) return DSPARK_ERR_INVALID_ARG;
    if (n > 0 && (!aligned16(ctr) || !aligned16(out))) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_philox_batch(ctr, keys, n, out, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_commit_lengths(const int32_t* n_accepted, const int32_t* l, int R, int gamma,
                          int32_t* commit_len, int32_t* cu_commit, int32_t* discard,
                          int32_t* total, int32_t* dev_status, dspark_stream_t stream) {
    if (!n_accepted || !commit_len || !cu_commit || !discard) return DSPARK_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || gamma > 16) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_commit(n_accepted, l, R, gamma, commit_len, cu_commit, discard,
                                     total, dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// draft_tc.cu -- Markov-head kernels on the tcgen05 tensor cores.
//
// "DSpark explainer" (papers.franksyz.com topic 31) sections 6-7 and llama.cpp
// PR 25173 (draft-dspark): per block position k the drafter's logits are
// U_k + W2 . W1[prev] with prev the anchor (k = 0) or the token drafted at
// k - 1, sampled left to right; the PR's "future work" asks for the bias and
// the argmax fused into one kernel, which is what one launch here is.
// Explainer sections 2-3: after the first rejection at position j the extra
// token comes from max(0, p - q) of row j; after full acceptance from p of the
// row after the block.
//
// One pipeline, two epilogues:
//   draft     one launch for the whole block: at each position k the logits of
//             every request, the Gumbel-max sample and the pieces of its
//             log-normaliser and q(y);
//   residual  one launch per verify: for every request the drafter's logits of
//             its rejected row are recomputed here (the residual needs q on the
//             whole vocabulary, and recomputing one row per request costs one
//             pass over W2 instead of keeping every drafted row in memory),
//             then the extra token is drawn from max(0, p - q), or from p after
//             full acceptance (the last CTA to finish writes the tokens).
//
// Persistent, one CTA per SM, 19 warps:
//   A (M = 128 requests x K = rank) = rows W1[prev] in tensor memory (columns
//     256-511, two bf16 per column), written by the epilogue threads with
//     tcgen05.st at the start of each step (prev: the anchor at k = 0, else the
//     step's predecessor decoded from the previous step's winner keys; the
//     residual: the rejected position's predecessor) and resident for the step,
//     so that shared memory is left to the W2 ring;
//   B (N = 128 vocabulary rows x K = rank) = W2 tiles streamed by TMA through a
//     ring of 16 KB stages (8, 128 KB in flight per SM; 6 to 12 measure alike,
//     4 is slower; no L2 prefetch ahead of the ring, which only added traffic);
//     the draft's W2 loads carry an L2 policy that keeps a fixed 30 % of W2's
//     lines resident from one position to the next (evict_last) and marks the
//     rest evict_first, and the U loads evict_first;
//   D = A . B^T in fp32 tensor memory, two 128-column buffers so the epilogue
//     of one vocabulary tile overlaps the MMAs of the next;
//   U_k (draft) = the tile's base logits, by TMA into two 16 KB pass buffers
//     (128 requests x 64 columns, 128-byte-swizzled) one pass ahead of the
//     epilogue, which adds them to the accumulator;
//   epilogue (16 warps; thread = one request x 32 vocabulary columns of a
//     tile, in two 16-column passes, pass h over columns 64 h .. 64 h + 63 of
//     the tile across the four warps of a lane quadrant).  Draft draws are
//     Gumbel-max with the noise built per 16-entry segment (one thread's pass
//     is one segment): the segments race in the exponential-race form (with
//     weight W = the segment's sum of exp and E = -log(u), the largest
//     log W + Gumbel(u) is the largest W / E, so a segment replaces the record
//     when W * E_best > W_best * E; since E >= 1 - u, a segment with
//     1 - u >= W * E_best / W_best cannot win, a test that needs no logarithm),
//     the record keeps its segment's logits in registers, and the entry is
//     picked once per step, from the record, by its running sum against a
//     second uniform times W.  The residual races entry by entry, with the
//     same no-log test, only the entries that pass it taking the logarithm
//     (a short series in 1 - u near u = 1, the special-function log2
//     elsewhere; relative error about 2e-6).  The four threads racing over a
//     request row in a CTA (one per quarter) share their best records through
//     shared memory, so each test uses the strongest of the four.
//   The residual launch also needs each request's own target row and U row
//     (128 scattered rows): six staging buffers, each one 32-column pass of
//     those rows, filled by the epilogue threads' own cp.async copies four
//     passes ahead; the epilogue works in four 32-column passes per tile, 8
//     columns per thread.
//
// Fused drafter logits (a third instantiation of the draft): the base logits
// are not given but formed in the same accumulator, U_k = W_lm . h_k with W_lm
// the lm_head the drafter shares with the target and h_k the backbone's hidden
// state at position k (explainer section 6; PR 25173 description), so one
// contraction over K = d + rank gives the whole logit:
//   s = [W_lm | W2] . [h_k ; W1[prev]].
// Each vocabulary tile first runs d / 64 k-blocks whose ring stage (32 KB)
// holds a W_lm block (B, TMA 2-D) and an h_k block (A, TMA 3-D, 128 requests
// x 64 hidden elements, read from L2 after the first tile), both from shared
// memory, then the rank / 64 W2 k-blocks with A = W1[prev] in tensor memory
// as above.  No U is read or written: the U producer idles and the epilogue
// takes the accumulator as the logit.  The MMA issuer waits for the step's A
// rows only before its first W2 k-block, so the first tile's lm_head part
// overlaps the hand-over between positions.
//
// Cross-CTA results need no merging pass: every CTA folds its winner into one
// 64-bit key per request and step with atomicMax (order-preserving bits of
// the score above the inverted index, so ties go to the lower index), and
// stores its (max, sum of exp, winner logit) piece of the normaliser.  The
// draft's steps run in one cooperative launch: after step k every CTA passes
// a grid barrier (a counter per step, bounded spin) and only then decodes the
// next A rows from the keys of step k.  Nothing else waits: the W2 ring and
// the U passes do not depend on the draws and stream on into the next step
// while the epilogue finishes the current one, and tensor memory, barriers
// and the ring are set up once per block instead of once per position.  After
// one more grid barrier past the last step, the epilogue warps of the grid
// turn keys and pieces into tokens, q_lse and q(y).
//
// Warp roles: warp 0 = W2 TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warp 2 = U TMA producer (draft), warps 3-18 = epilogue (and the A
// rows).  The three control warps each share a scheduler with four epilogue
// warps that leave them few issue slots, so each runs its loop as a whole warp
// (its state in uniform registers) and lets one elected lane issue the copies,
// MMAs and commits.  Every mbarrier wait and the grid barrier are bounded
// (2 s); a timeout aborts every CTA cleanly and reports DSPARK_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_fp16.h>

#include "draft_tc.cuh"
#include "tc_ptx.cuh"

namespace dspark {
namespace {

constexpr int kM = 128;                       // requests per CTA (MMA M)
constexpr int kNV = 128;                      // vocabulary rows per tile (MMA N)
constexpr int kKB = 64;                       // rank elements per stage (128-byte rows)
constexpr int kTileBytes = 128 * kKB * 2;     // 16 KB: one operand k-block
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kCtlWarps = 3;                  // W2 producer, MMA issuer, U producer
constexpr int kThreads = kCtlWarps * 32 + kEpiThreads;
constexpr int kPassCols = 16;                 // of which one pass handles
constexpr int kUBufBytes = kM * 64 * 2;       // base logits of one pass: 128 requests x 64 columns
constexpr int kUBufs = 2;                     // draft: pass buffers of base logits (one tile)
// residual staging of one 32-column pass for the 128 requests: target logits
// (fp32, 128-byte rows) and base logits (bf16, 64-byte rows), copied in
// 16-byte pieces by the epilogue threads a few passes ahead
constexpr int kResCols = 32;
constexpr int kResTBytes = kM * kResCols * 4;  // 16 KB
constexpr int kResUBytes = kM * kResCols * 2;  // 8 KB
constexpr int kResBufs = 6;                    // staging buffers
constexpr int kResAhead = kResBufs - 2;        // passes whose copies are issued ahead of the one computed
constexpr int kMaxStages = 8;
constexpr int kMaxKb = 8;                   // k-blocks of a tile at rank 512, the largest
constexpr int kMaxP = 256;                    // CTAs per request block (pieces per request)
constexpr uint32_t kTmemCols = 512;     // two 128-column accumulators, then the A rows (at most 256 columns)
constexpr uint32_t kAcol = 256;         // first tensor-memory column of A
constexpr uint64_t kWaitNs = 2000000000ull;
// The draft's W2 loads keep this fraction of W2's lines resident in L2 from one
// position to the next (the same lines every time; the rest, and every U load,
// are first to be evicted): W2 is larger than L2, so plain LRU keeps none of it.
// At the R = 128 bench shape 0.2, 0.3 and 0.4 measured 261.4, 261.1 and 262.3 us
// per draft call, 0.6 272 us, and no hints 273.3 us.
constexpr float kW2KeepFraction = 0.3f;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
// Relative slack of the no-log race test, far above the rounding of the
// quantities it compares (a few units in 2^-24).
constexpr float kRaceSlack = 1.0f + 0x1p-10f;

// Per-request partial of one thread or CTA.  Draft: (score, idx) of the
// Gumbel-max draw, s at it, (max, sum of exp) of the logits.  Residual:
// (score, idx) of the draw.
struct TcPartial {
    float score;
    int idx;
    float s_at;
    float m, sum;
    float pad[3];
};
// the draft's end-of-step exchange of the epilogue quarters ([3][kM]), whole KB
constexpr int kExchBytes = (3 * kM * (int)sizeof(TcPartial) + 1023) / 1024 * 1024;


struct TcParams {
    const uint16_t* U;
    const uint16_t* W1;
    int w1_wide;               // W1 is 32-byte aligned: its rows are read 32 bytes a lane at a time
    unsigned long long* keys;  // draft [gamma][R]; residual [R]
    unsigned* step_done;       // draft [gamma]: CTAs done with step k; then one abort word
    float4* parts;             // draft [gamma][R][P]: (max, sum, winner logit, winner) per CTA
    const uint64_t* seeds;
    int32_t* dev_status;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank;
    int nb, P, n_tiles, n_stages, nkb;
    int dkb;                   // fused drafter logits: 64-element k-blocks of the hidden size (else 0)
    const int32_t* anchor;
    float* q_logits;
    int32_t* y;                // draft outputs [R][gamma]
    float* q_lse;
    float* q_tok;
    const float* target;
    const ResRow* rows;
    int32_t* out_tokens;       // residual: [R][gamma + 1]
    // draft: the grid barriers between positions wait at most wait_ns; their
    // arrival count is the grid's plus phantom (1 only in the timeout test)
    unsigned long long wait_ns;
    unsigned phantom;
};

struct Bars {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t tfull[2], tempty[2];
    uint64_t ufull[kUBufs], uempty[kUBufs];
    uint64_t sfull[kResBufs], sempty[kResBufs];  // residual staging buffers
    uint64_t afull, mma_done;  // afull: the step's A rows are in shared memory (one arrival per epilogue warp)
    uint32_t tmem_slot;
    int abort_flag;
    int step_ok;               // the grid barrier after a step passed (read by every epilogue warp)
    int fin_last, fin_nfb;     // residual tokens: this CTA is the last one done; requests drawn from p
    unsigned long long fin_key;
    int a_tok[kM];             // the step's A rows' tokens: -1 zero row, -2 nothing to compute for the request
};
// Residual-only shared memory after the barriers: per request row and epilogue
// quarter the best race record so far as log2(w / E) in absolute units (-inf:
// none), read by the row's other quarters; then each request's target row and
// U row (-1 when not needed), from which every epilogue thread takes the rows
// of its staging copies.
struct ResShared {
    float g_share[4][kM];
    int trow[kM];
    int urow[kM];
};
constexpr size_t kShareBytes = sizeof(ResShared);
// Draft-only shared memory after the barriers: per request row, the best race
// record of each epilogue quarter as G = log2(w / E) in absolute base-2 units
// (the record's scaled logit minus log2 E), rounded down to half precision: a
// smaller G is a looser bound, so still a valid one; -inf when none yet.
struct DraftShared {
    __half g[kM][4];
};

__device__ __forceinline__ void merge_draft(float& sc, int& ix, float& sa, float& m, float& su, float sc2, int ix2,
                                            float sa2, float m2, float su2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; sa = sa2; }
    lse_merge(m, su, m2, su2);
}

template <bool kRes>
__device__ __forceinline__ void merge_any(TcPartial& a, const TcPartial& b) {
    if (kRes) {
        if (better(b.score, b.idx, a.score, a.idx)) { a.score = b.score; a.idx = b.idx; }
    } else {
        merge_draft(a.score, a.idx, a.s_at, a.m, a.sum, b.score, b.idx, b.s_at, b.m, b.sum);
    }
}

template <bool kRes>
__device__ __forceinline__ TcPartial identity_partial() {
    TcPartial w;
    w.score = -INFINITY; w.idx = INT_MAX; w.s_at = 0.0f;
    w.m = -INFINITY; w.sum = 0.0f;
    w.pad[0] = w.pad[1] = w.pad[2] = 0.0f;
    return w;
}

// (score, idx) as one integer whose unsigned order is better()'s order: the
// score's bits made order-preserving (negative floats inverted, positive ones
// with the sign bit set; -0 folded onto +0) above the inverted index.  A
// published key is never 0.
__device__ __forceinline__ unsigned long long winner_key(float score, int idx) {
    uint32_t b = __float_as_uint(score + 0.0f);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (unsigned long long)(~(uint32_t)idx);
}

__device__ __forceinline__ int key_index(unsigned long long key) { return (int)~(uint32_t)key; }

// Vocabulary tile of a CTA's launch-global tile g (step g / n_local, the
// step's i-th tile of the CTA's tiles cidx, cidx + P, ...).  (Running odd steps
// in reverse order, to start on tiles still in L2, measured slower.)
__device__ __forceinline__ int tile_at(int g, int n_local, int cidx, int P) {
    return cidx + (g % n_local) * P;
}

// 2^x on the special-function unit (relative error about 2^-22; the race
// decisions and normalisers it feeds carry far larger margins).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// E_best / w_best with the slack of the no-log test.  An approximate quotient
// (a few units in 2^-24) is far inside the 2^-10 slack; w_best = 0 gives +inf
// (every entry with w > 0 is then a candidate).
__device__ __forceinline__ float race_bound(float e_best, float w_best) {
    return __fdividef(e_best, w_best) * kRaceSlack;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2 of the ratio w / E encoded in a published winner key (natural-log
// score in the high word); -inf when nothing is published yet.
__device__ __forceinline__ float key_log2_ratio(unsigned long long key) {
    if (key == 0) return -INFINITY;
    const uint32_t hi = (uint32_t)(key >> 32);
    const uint32_t bits = (hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi;
    return __uint_as_float(bits) * kLog2eF;
}

// 1 + (1 - u) - 2^-24 for u = uniform_from_bits(x): the 23 kept bits inverted
// under the exponent of 1.0 (exact).
__device__ __forceinline__ float one_plus_complement(uint32_t x) {
    return __uint_as_float((x >> 9) ^ 0x3FFFFFFFu);
}

// E = -ln(u) for u = uniform_from_bits(x), with relative error below about
// 2e-6, without a branch: for u near 1 from d = 1 - u (exact from the bits) by
// the series d + d^2/2 + ... + d^5/5 (truncation below d^5 / 6 relative for
// d < 1/16), else from the special-function unit's log2 (absolute error about
// 2^-22 on |log2 u| >= 0.09).
__device__ __forceinline__ float neg_log_uniform(uint32_t x) {
    const float d = (__uint_as_float((x >> 9) ^ 0x3FFFFFFFu) - 1.0f) + 0x1p-24f;
    const float series = d * fmaf(d, fmaf(d, fmaf(d, fmaf(d, 0.2f, 0.25f), 1.0f / 3.0f), 0.5f), 1.0f);
    float l2;
    asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(uniform_from_bits(x)));
    return d < 0.0625f ? series : -l2 * kLn2F;
}

// a[c] for a register array of N (a power of two) and a lane-varying c in
// [0, N): a tree of selects on the bits of c, lowest bit first (register
// arrays cannot be indexed at run time without a trip through local memory)
template <int N, typename T>
__device__ __forceinline__ T pick(const T (&a)[N], int c) {
    T l[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) l[i] = (c & 1) ? a[2 * i + 1] : a[2 * i];
    if constexpr (N == 2)
        return l[0];
    else
        return pick<N / 2>(l, c >> 1);
}

__device__ __forceinline__ uint32_t word_of(const uint4& x, int j) {
    return j == 0 ? x.x : (j == 1 ? x.y : (j == 2 ? x.z : x.w));
}

// 32 bytes at p (32-byte aligned, read-only for the kernel's lifetime) in one load.
__device__ __forceinline__ void ldg_nc_32b(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// 16 bytes global -> shared without registers; zeros when !valid (nothing read).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// One arrival on bar once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// The 16 epilogue warps alone (named barrier 1; barrier 0 is the CTA's).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

// Between two draft steps, one thread per CTA: every CTA's winner keys of the
// step are published (its threads passed a CTA barrier after their atomics)
// before any CTA reads them.  done counts the CTAs through the step (zeroed
// with the keys before the launch, used once).  Bounded: gives up after
// wait_ns or when another CTA gave up (abort word), raising the abort word
// itself on a timeout.
__device__ __forceinline__ bool step_barrier(unsigned* done, int* abort_word, unsigned n_cta,
                                             unsigned long long wait_ns) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(done) : "memory");
    const uint64_t t0 = global_ns();
    for (unsigned it = 1;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(done) : "memory");
        if (v >= n_cta) break;
        if ((it & 15) == 0) {
            if (*reinterpret_cast<volatile int*>(abort_word)) return false;
            if (global_ns() - t0 > wait_ns) {
                atomicExch(abort_word, 1);
                return false;
            }
        }
    }
    return true;
}


// Residual launch, after every CTA has published its winner keys: the last
// CTA to finish writes every request's extra token -- the race's winner, or,
// when a rejected row's residual had no positive mass (p <= q everywhere, a
// rounding-level event), a draw from p of the row with the same noise, made by
// the whole CTA.  The dynamic shared memory is free by then and holds the list
// of those requests.  keys[R] counts the CTAs that are done (zeroed with the
// keys by the verify prologue).
__device__ void residual_tokens_if_last(const TcParams& p, uint8_t* smem, Bars& bar) {
    int& s_last = bar.fin_last;
    int& s_nfb = bar.fin_nfb;
    unsigned long long& s_key = bar.fin_key;
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's keys before its count
        s_last = atomicAdd(p.keys + p.R, 1ull) == (unsigned long long)(gridDim.x - 1);
        s_nfb = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // every CTA's keys (their counts came first)
    int* fb = reinterpret_cast<int*>(smem);
    const int g1 = p.gamma + 1;
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {  // one request per thread
        const int mode = p.rows[r].mode, pos = p.rows[r].pos;
        const unsigned long long key = __ldcg(p.keys + r);
        if (mode == 0) continue;
        if (key == 0 && mode == 1) {
            fb[atomicAdd(&s_nfb, 1)] = r;
            continue;
        }
        const int tok = key ? key_index(key) : -1;
        if (tok < 0) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);  // no finite score (NaN logits)
        p.out_tokens[(size_t)r * g1 + pos] = tok;
    }
    __syncthreads();
    const float c2 = p.invT * kLog2eF;
    for (int i = 0; i < s_nfb; ++i) {
        const int r = fb[i];
        const ResRow ri = p.rows[r];
        if (threadIdx.x == 0) s_key = 0;
        __syncthreads();
        const float* trow = p.target + (size_t)ri.trow * p.V;
        const uint64_t seed = p.seeds[r];
        float bw = 0.0f, bE = 1.0f;
        int bi = INT_MAX;
        for (int v4 = threadIdx.x; 4 * v4 < p.V; v4 += blockDim.x) {
            const uint4 x = philox4x32_10(make_uint4((uint32_t)v4, (uint32_t)ri.pos, (uint32_t)r, ri.w3),
                                          (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 4 * v4 + e;
                if (v >= p.V) break;
                const float pv = ex2(fmaf(__ldg(trow + v), c2, -ri.lse2_p));
                const float E = neg_log_uniform(word_of(x, e));
                if (pv * bE > bw * E) { bw = pv; bE = E; bi = v; }
            }
        }
        if (bi != INT_MAX) atomicMax(&s_key, winner_key(logf(bw) - logf(bE), bi));
        __syncthreads();
        if (threadIdx.x == 0) {
            const int tok = s_key ? key_index(s_key) : -1;
            if (tok < 0) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
            p.out_tokens[(size_t)r * g1 + ri.pos] = tok;
        }
        __syncthreads();
    }
}

// tm_u: U [R, gamma, V] (draft), or for the fused draft the hidden states h
// [R, gamma, d] (the same box: 64 elements x 1 position x 128 requests);
// tm_wlm: the fused draft's lm_head [V, d] (unused otherwise).
template <bool kRes, bool kFused = false>
__global__ void __launch_bounds__(kThreads, 1)
markov_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
                 const __grid_constant__ CUtensorMap tm_wlm, const TcParams p) {
    static_assert(!(kRes && kFused), "the residual recomputes from given base logits");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // A lives in tensor memory.  Draft: quarter exchange | two U pass buffers |
    // W2 ring; residual: target staging buffers | base-logit staging buffers |
    // W2 ring
    uint8_t* sX = smem;
    uint8_t* sU = kRes ? smem : sX + kExchBytes;
    uint8_t* sRT = sU;
    uint8_t* sRU = sU + kResBufs * kResTBytes;
    // fused: no U pass buffers; a ring stage holds B (W_lm or W2 block) then A (h block)
    constexpr int kStage = kFused ? 2 * kTileBytes : kTileBytes;
    uint8_t* sB = sU + (kRes ? kResBufs * (kResTBytes + kResUBytes) : (kFused ? 0 : kUBufs * kUBufBytes));
    Bars& bar = *reinterpret_cast<Bars*>(sB + p.n_stages * kStage);
    ResShared& rsh = *reinterpret_cast<ResShared*>(&bar + 1);  // residual only
    DraftShared& dsh = *reinterpret_cast<DraftShared*>(&bar + 1);  // draft only
    float* g_share = &rsh.g_share[0][0];
    // the quarters' exchange at the end of a step ([3][kM]): draft, its own
    // space (the ring and the U buffers stream on into the next step);
    // residual, the W2 ring (drained when the last tile's accumulator has been
    // seen)
    TcPartial* scratch = reinterpret_cast<TcPartial*>(kRes ? sB : sX);
    volatile int* abort_flag = &bar.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = blockIdx.x % p.nb;
    const int cidx = blockIdx.x / p.nb;
    const int row0 = blk * kM;
    const int S = p.n_stages;
    const int n_steps = kRes ? 1 : p.gamma;

    if (kRes)
        for (int e = threadIdx.x; e < 4 * kM; e += kThreads) g_share[e] = -INFINITY;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { tc::mbar_init(&bar.full[s], 1); tc::mbar_init(&bar.empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar.tfull[a], 1); tc::mbar_init(&bar.tempty[a], kEpiWarps); }
        for (int a = 0; a < kUBufs; ++a) { tc::mbar_init(&bar.ufull[a], 1); tc::mbar_init(&bar.uempty[a], kEpiWarps); }
        for (int a = 0; a < kResBufs; ++a) {
            tc::mbar_init(&bar.sfull[a], kEpiThreads);  // one cp.async arrival per epilogue thread
            tc::mbar_init(&bar.sempty[a], kEpiWarps);
        }
        tc::mbar_init(&bar.afull, kEpiWarps);
        tc::mbar_init(&bar.mma_done, 1);
        bar.abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bar.tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tm_w2);
        if (!kRes) tc::prefetch_tmap(&tm_u);
        if (kFused) tc::prefetch_tmap(&tm_wlm);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = bar.tmem_slot;
    const int n_local = cidx < p.n_tiles ? (p.n_tiles - 1 - cidx) / p.P + 1 : 0;
    const int n_tl = n_steps * n_local;  // tiles of this CTA over the launch: step-major

    // this thread's running partial (epilogue threads)
    TcPartial part = identity_partial<kRes>();
    bool row_ok = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The W2 ring, tile-major over every step of the launch (the tiles are the
        // same at each step): nothing here depends on the draws, so the ring runs
        // into the next step while the epilogue finishes the current one.  (No L2
        // prefetch ahead of the ring: the deep ring alone keeps HBM streaming, and
        // prefetch requests measured as extra traffic that slowed it.)  The whole
        // warp runs the loop and one elected lane issues each load.  With several
        // request blocks (their CTAs reread each tile from L2) the loads must go out
        // as soon as stages free: the indices are counters, and this form took the
        // R = 512 draft from 0.52 to 0.37 ms against a lane-0 loop that divides per
        // load.  With one block (every tile streamed from HBM once) the dividing
        // loop measured 2-4 % faster at R = 128 with sampling (and as much slower
        // at R = 16 greedy); no load order or issue pacing that was tried explains
        // it, and it is kept for that case.
        const uint64_t pol_w2 = tc::policy_keep_fraction(kW2KeepFraction);  // the draft's W2 (see above)
        const int n_loads = n_tl * (p.dkb + p.nkb);  // stage loads
        int issued = 0;
        bool ok = true;
        if constexpr (kFused) {
            // per tile: d / 64 stages of (W_lm block, h block of the tile's step), then
            // rank / 64 W2 stages; the same counters as below plus the step
            const int nkt = p.dkb + p.nkb;
            int s = 0, kb = 0, i = 0, t = cidx, step = 0;  // stage, k-block, local tile, tile, step
            uint32_t ph = 0;
            for (; issued < n_loads; ++issued) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                uint8_t* st = sB + s * kStage;
                if (kb < p.dkb)
                    tc::tma_load_2d_3d_elect(st, &tm_wlm, kb * kKB, t * kNV, st + kTileBytes, &tm_u, kb * kKB, step,
                                             row0, &bar.full[s], 2u * kTileBytes);
                else
                    tc::tma_load_2d_elect(st, &tm_w2, &bar.full[s], (kb - p.dkb) * kKB, t * kNV, kTileBytes);
                if (++s == S) { s = 0; ph ^= 1u; }
                if (++kb == nkt) {
                    kb = 0;
                    if (++i == n_local) { i = 0; t = cidx; ++step; } else { t += p.P; }
                }
            }
        } else if (p.nb == 1) {
            for (; issued < n_loads; ++issued) {
                // load l goes to stage l % S, used for the (l / S)-th time
                const int s = issued % S;
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                const int g = issued / p.nkb, kb = issued - g * p.nkb;
                const int t = tile_at(g, n_local, cidx, p.P);
                if (!kRes)
                    tc::tma_load_2d_elect_hint(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV, kTileBytes,
                                               pol_w2);
                else
                    tc::tma_load_2d_elect(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV, kTileBytes);
            }
        } else {
            int s = 0, kb = 0, i = 0, t = cidx;  // stage, k-block, local tile, tile
            uint32_t ph = 0;
            for (; issued < n_loads; ++issued) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                if (!kRes)
                    tc::tma_load_2d_elect_hint(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV, kTileBytes,
                                               pol_w2);
                else
                    tc::tma_load_2d_elect(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV, kTileBytes);
                if (++s == S) { s = 0; ph ^= 1u; }
                if (++kb == p.nkb) {
                    kb = 0;
                    if (++i == n_local) { i = 0; t = cidx; } else { t += p.P; }
                }
            }
        }
        // the copies this warp issued must land before the CTA exits
        if (!ok && lane == 0) {
            int dummy = 0;
            volatile int* no_abort = &dummy;
            for (int l = max(0, issued - S); l < issued; ++l)
                tc::mbar_wait(&bar.full[l % S], (uint32_t)((l / S) & 1), no_abort, kWaitNs);
        }
        __syncwarp();  // the warp reconverges before the CTA-wide barrier below
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop and waits; one elected lane issues the MMAs
        // and commits (a lane-0 loop cost about 100 cycles of issue per MMA with
        // the epilogue idle and ~180 beside a busy one, against 64 for the MMA).
        // A tile's k-block kb reads A from column kAcol + 32 kb and B from ring
        // stage s, whose descriptor is the ring base's plus s * 16 KB.
        constexpr uint32_t idesc = tc::idesc_bf16_f32(kM, kNV);
        bool ok = true;
        int s = 0;
        uint32_t ph = 0;
        const uint64_t desc0 = tc::smem_desc_sw128(tc::smem_u32(sB));
        const uint32_t a_base = tmem_base + kAcol;
        for (int k = 0; ok && k < n_steps; ++k) {
            // the step's A rows, written by the epilogue warps (fused: awaited before
            // the first W2 k-block of the step, below)
            if (!kFused) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.afull, (uint32_t)(k & 1), abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
            }
            for (int i = 0; ok && i < n_local; ++i) {
                const int g = k * n_local + i;
                const int a = g & 1;
                const uint32_t use = (uint32_t)(g >> 1);
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.tempty[a], (use & 1u) ^ 1u, abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kNV);
                if constexpr (kFused) {
                    // the lm_head part: A (h block) and B (W_lm block) both in the stage
#pragma unroll 1
                    for (int kb = 0; kb < p.dkb; ++kb) {
                        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.full[s], ph, abort_flag, kWaitNs))) {
                            ok = false;
                            break;
                        }
                        tc::tc_fence_after();
                        const uint64_t bd = desc0 + (uint64_t)(s * (kStage >> 4));
                        const uint64_t ad = bd + (uint64_t)(kTileBytes >> 4);
#pragma unroll
                        for (int j = 0; j < kKB / 16; ++j)
                            tc::umma_bf16_elect(d, ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j), idesc, (kb | j) != 0);
                        tc::umma_commit_elect(&bar.empty[s]);
                        if (++s == S) { s = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    if (i == 0) {  // from here on the step's A rows are read
                        if (!__all_sync(0xFFFFFFFFu,
                                        tc::mbar_wait(&bar.afull, (uint32_t)(k & 1), abort_flag, kWaitNs))) {
                            ok = false;
                            break;
                        }
                        tc::tc_fence_after();
                    }
                }
#pragma unroll
                for (int kb = 0; kb < kMaxKb; ++kb) {
                    if (kb < p.nkb) {  // warp-uniform
                        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.full[s], ph, abort_flag, kWaitNs))) {
                            ok = false;
                            break;
                        }
                        tc::tc_fence_after();
                        const uint64_t bd = desc0 + (uint64_t)(s * (kStage >> 4));
#pragma unroll
                        for (int j = 0; j < kKB / 16; ++j)  // A: K elements 64 kb + 16 j .. at column 32 kb + 8 j
                            tc::umma_bf16_ta_elect(d, a_base + (uint32_t)(32 * kb + 8 * j), bd + (uint64_t)(2 * j),
                                                   idesc, kFused || (kb | j) != 0);
                        tc::umma_commit_elect(&bar.empty[s]);
                        if (++s == S) { s = 0; ph ^= 1u; }
                    }
                }
                if (ok) tc::umma_commit_elect(&bar.tfull[a]);
            }
        }
        // every MMA issued has completed before anyone frees tensor memory
        tc::umma_commit_elect(&bar.mma_done);
        int dummy = 0;
        volatile int* no_abort = &dummy;
        tc::mbar_wait(&bar.mma_done, 0, no_abort, kWaitNs);
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ U producer
        // Draft: the base logits U_k of pass n (global tile n / 2, columns 64 (n % 2)
        // .. + 63 of the tile, all 128 requests) into pass buffer n % kUBufs, up to
        // kUBufs passes ahead of the epilogue, across the steps of the launch
        // (deeper buffering measured no faster: the W2 ring is what bounds a tile).
        if (!kRes && !kFused) {
            const int n_pass = 2 * n_tl;
            const uint64_t pol_u = tc::policy_evict_first();  // each U_k is read once
            int n = 0;
            int b = 0, half = 0, i = 0, step = 0, t = cidx;  // buffer, pass of the tile, local tile, step, tile
            uint32_t uph = 0;
            for (; n < n_pass; ++n) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.uempty[b], uph ^ 1u, abort_flag, kWaitNs))) break;
                tc::tma_load_3d_elect_hint(sU + b * kUBufBytes, &tm_u, &bar.ufull[b], t * kNV + 64 * half, step, row0,
                                           (uint32_t)kUBufBytes, pol_u);
                if (++b == kUBufs) { b = 0; uph ^= 1u; }
                if (++half == 2) {
                    half = 0;
                    if (++i == n_local) { i = 0; t = cidx; ++step; } else { t += p.P; }
                }
            }
            // the copies this warp issued must land before the CTA exits
            if (lane == 0) {
                int dummy = 0;
                volatile int* no_abort = &dummy;
                for (int l = max(0, n - kUBufs); l < n; ++l)
                    tc::mbar_wait(&bar.ufull[l % kUBufs], (uint32_t)((l / kUBufs) & 1), no_abort, kWaitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = threadIdx.x - kCtlWarps * 32;  // 0..511
        const int ew = warp - kCtlWarps;   // 0..15
        const int quad = warp & 3;         // TMEM lane quadrant this warp may read
        const int quarter = ew >> 2;       // pass h covers columns 64 h + 16 quarter .. + 15 of a tile
        const int m = quad * 32 + lane;
        const int rr = row0 + m;
        ResRow rinfo;
        rinfo.mode = 0; rinfo.pos = 0; rinfo.trow = 0; rinfo.w3 = 0; rinfo.lse2_p = 0.0f; rinfo.q_lse2 = 0.0f;
        if (kRes && rr < p.R) rinfo = p.rows[rr];
        const bool sampling = kRes || !p.greedy;
        const uint64_t seed = (sampling && rr < p.R) ? p.seeds[rr] : 0ull;
        const uint32_t key0 = (uint32_t)(seed & 0xFFFFFFFFu), key1 = (uint32_t)(seed >> 32);
        const uint32_t w3 = kRes ? rinfo.w3 : ctr_word3(p.cycle, kDraftGumbel);
        const bool with_u = !kRes || rinfo.mode == 1;
        // logits are scaled to base 2 when sampling: s2 = s * log2(e) / T
        const float c2 = sampling ? p.invT * kLog2eF : 1.0f;
        // draft: this thread's 32 bytes of a pass buffer (row m, 16-byte chunks
        // 2 quarter and 2 quarter + 1 of the 128-byte-swizzled row)
        const uint32_t u_off0 = (uint32_t)(m * 128 + (((2 * quarter) ^ (m & 7)) << 4));
        const uint32_t u_off1 = (uint32_t)(m * 128 + (((2 * quarter + 1) ^ (m & 7)) << 4));
        const int cpr = p.rank >> 3;  // 16-byte pieces of a W1 row (at most 64)

        for (int k = 0; k < n_steps; ++k) {
            // no race record of this step yet (the previous step's readers are past
            // the barriers at its end; this step's read after the one below)
            if (!kRes) *reinterpret_cast<volatile unsigned short*>(&dsh.g[m][quarter]) = 0xFC00u;
            // ---- the step's A rows: tokens (the anchor at k = 0, else the previous
            // step's winner, decoded from its key; residual: the rejected
            // position's predecessor), then W1 rows: draft, into the 128-byte-
            // swizzled K-major layout the MMA descriptors describe (16-byte piece c
            // of row j at k-block c / 8, row j, piece (c % 8) ^ (j % 8)); residual,
            // into tensor memory
            if (e < kM) {
                const int r = row0 + e;
                int t = -2;
                if (r < p.R) {
                    if constexpr (kRes) {
                        const ResRow& rw = p.rows[r];
                        t = rw.mode == 0 ? -2 : rw.prev;
                        rsh.trow[e] = rw.mode != 0 ? rw.trow : -1;
                        rsh.urow[e] = rw.mode == 1 ? r * p.gamma + rw.pos : -1;
                    } else if (k == 0) {
                        const int an = p.anchor[r];
                        t = an >= p.V ? -2 : (an < 0 ? -1 : an);
                    } else {
                        // published by every CTA's atomics before the step barrier: read from L2
                        const unsigned long long key = __ldcg(p.keys + (size_t)(k - 1) * p.R + r);
                        t = key ? key_index(key) : -2;
                    }
                }
                bar.a_tok[e] = t;
                if (kRes && r >= p.R) { rsh.trow[e] = -1; rsh.urow[e] = -1; }
            }
            epi_sync();
            // Residual staging: thread e copies target pieces e and e + 512 (piece c of
            // row m: c = piece % 8, m = piece / 8) and base-logit piece e (c = e % 4,
            // m = e / 4) of every pass, so that one warp instruction moves four whole
            // 128-byte target rows or eight 64-byte U rows; pieces past the row end,
            // and rows without a draw, are zero-filled without a read.  The copies
            // of pass n go out kResAhead passes before it is computed.
            const int n_res = kRes ? 4 * n_local : 0;
            const int stc = e & 7, stm0 = e >> 3, stm1 = stm0 + 64, suc = e & 3, sum_ = e >> 2;
            const int st_t0 = kRes ? rsh.trow[stm0] : -1, st_t1 = kRes ? rsh.trow[stm1] : -1;
            const int st_u = kRes ? rsh.urow[sum_] : -1;
            const uint32_t st_d0 = (uint32_t)(stm0 * 128 + ((stc ^ (stm0 & 7)) << 4));
            const uint32_t st_d1 = (uint32_t)(stm1 * 128 + ((stc ^ (stm1 & 7)) << 4));
            const uint32_t st_du = (uint32_t)(sum_ * 64 + ((suc ^ ((sum_ >> 1) & 3)) << 4));
            // false when the wait for a free buffer gave up
            auto stage_issue = [&](int n) -> bool {
                const int b = n % kResBufs;
                const uint32_t use = (uint32_t)(n / kResBufs);
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.sempty[b], (use & 1u) ^ 1u, abort_flag, kWaitNs)))
                    return false;
                const int v = (cidx + (n >> 2) * p.P) * kNV + kResCols * (n & 3);
                const int ct = v + 4 * stc, cu = v + 8 * suc;
                const bool i0 = st_t0 >= 0 && ct < p.V, i1 = st_t1 >= 0 && ct < p.V, iu = st_u >= 0 && cu < p.V;
                cp_async_16(sRT + b * kResTBytes + st_d0, p.target + (i0 ? (size_t)st_t0 * p.V + ct : 0), i0);
                cp_async_16(sRT + b * kResTBytes + st_d1, p.target + (i1 ? (size_t)st_t1 * p.V + ct : 0), i1);
                cp_async_16(sRU + b * kResUBytes + st_du, p.U + (iu ? (size_t)st_u * p.V + cu : 0), iu);
                cp_async_arrive(&bar.sfull[b]);
                return true;
            };
            bool staged = true;
            if constexpr (kRes) {
                // residual: A in tensor memory from column kAcol (lane = request row,
                // two bf16 per column).  The rows first pass through the staging
                // buffers (not in use yet): warp ew copies rows 8 ew .. 8 ew + 7 whole
                // with cp.async (16-byte piece c of row j at j * rank * 2 +
                // (c ^ (j % 8)) * 16, zeros for a negative token), so that each
                // warp instruction reads one row; then thread (row m, quarter) moves
                // row m's K elements rank/4 * quarter .. + rank/4 - 1 into tensor
                // memory, eight columns per store, its 32 rows' pieces on distinct banks.
                const int rowb = p.rank * 2;
#pragma unroll 1
                for (int q = 0; q < 8; ++q) {
                    const int j = 8 * ew + q;
                    const int t = bar.a_tok[j];
                    const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)(t < 0 ? 0 : t) * p.rank);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = lane + 32 * h;
                        if (c < cpr) cp_async_16(sRT + j * rowb + ((c ^ (j & 7)) << 4), src + c, t >= 0);
                    }
                }
                cp_async_wait_all();
                epi_sync();
                const int n16 = cpr >> 2;  // 16-byte pieces of a quarter row (at most 16)
                const uint32_t tq =
                    tmem_base + ((uint32_t)(quad * 32) << 16) + kAcol + (uint32_t)(quarter * (n16 * 4));
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    if (c < n16) {  // warp-uniform
                        const int pc = quarter * n16 + c;
                        const uint4 v0 = *reinterpret_cast<const uint4*>(sRT + m * rowb + ((pc ^ (m & 7)) << 4));
                        const uint4 v1 = *reinterpret_cast<const uint4*>(sRT + m * rowb + (((pc + 1) ^ (m & 7)) << 4));
                        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                        tc::tmem_st_32x32b_x8(tq + (uint32_t)(4 * c), w);
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bar.afull);
                // every thread has read its A pieces before the staging copies reuse the space
                epi_sync();
                for (int n = 0; staged && n < kResAhead && n < n_res; ++n) staged = stage_issue(n);
            } else {
                // draft: thread (row m, quarter) moves row m's K elements rank/4 *
                // quarter .. + rank/4 - 1 of W1[token] from global memory into tensor
                // memory (zeros for a negative token), every piece in flight at once
                const int n16 = cpr >> 2;  // 16-byte pieces of a quarter row (at most 16)
                const int tk0 = bar.a_tok[m];
                const int tk = (tk0 < 0 || IN_BOUNDS(tk0 < p.V, p.dev_status)) ? tk0 : -1;
                const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)(tk < 0 ? 0 : tk) * p.rank) +
                                   quarter * n16;
                const uint32_t tq =
                    tmem_base + ((uint32_t)(quad * 32) << 16) + kAcol + (uint32_t)(quarter * (n16 * 4));
                if (p.w1_wide) {  // warp-uniform: 32 bytes a lane per load, half the requests
                    uint32_t v[8][8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        if (2 * c < n16 && tk >= 0) {
                            ldg_nc_32b(src + 2 * c, v[c]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j) v[c][j] = 0u;
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        if (2 * c < n16) tc::tmem_st_32x32b_x8(tq + (uint32_t)(8 * c), v[c]);  // warp-uniform
                } else {
                    uint4 v[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        v[c] = (c < n16 && tk >= 0) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        if (c < n16) {  // warp-uniform
                            const uint32_t w[8] = {v[c].x, v[c].y, v[c].z, v[c].w,
                                                   v[c + 1].x, v[c + 1].y, v[c + 1].z, v[c + 1].w};
                            tc::tmem_st_32x32b_x8(tq + (uint32_t)(4 * c), w);
                        }
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bar.afull);
            }
            row_ok = rr < p.R && bar.a_tok[m] != -2;
            if (kRes) row_ok = row_ok && rinfo.mode != 0;
            const int pos = kRes ? rinfo.pos : k;
            const size_t rk = (size_t)rr * p.gamma + pos;
            float* qrow = (!kRes && p.q_logits && row_ok) ? p.q_logits + rk * p.V : nullptr;
            part = identity_partial<kRes>();
            // exponential-race state (bw, bE) and rho = E_best / w_best with the
            // slack, the bound of the no-log test.  Residual: an entry that cannot
            // beat the best record of any thread racing over the same request
            // cannot be the request's winner either, so rho is taken from the best
            // of this thread's record, the row's other three quarters in this CTA
            // (shared memory, every pass) and the request's published key (global,
            // read a tile late), each as g = log2(w / E) in absolute units.  (The
            // draft's races gain too little from this to pay for the atomics.)
            float bw = 0.0f, bE = 1.0f;
            float rho = INFINITY;
            // draft: the record segment's logits (before the temperature), its pick
            // word and first entry; the tile's segment words
            float seg[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) seg[c] = -INFINITY;
            uint32_t seg_a = 0u;
            int seg_v0 = 0;
            uint4 seg_words = make_uint4(0u, 0u, 0u, 0u);
            float g_own = -INFINITY, g_pub = -INFINITY, g_glob = -INFINITY;
            unsigned long long gkey = 0;
            const bool share = kRes && row_ok;
            unsigned long long* my_key = kRes ? p.keys + rr : p.keys + (size_t)k * p.R + rr;
            volatile float* gsh = g_share + m;  // the row's four quarter records, written by other warps
            if constexpr (!kRes) {
            // ---- draft: thread = request row m x 32 columns of a tile, two
            // 16-column passes (pass h covers columns 64 h + 16 quarter .. + 15)
            for (int i = 0; i < n_local; ++i) {
                const int g = k * n_local + i;  // global tile of the launch: TMEM buffer, U pass phases
                const int t = tile_at(g, n_local, cidx, p.P);
                const int a = g & 1;
                const uint32_t use = (uint32_t)(g >> 1);
                // warp-uniform wait: every lane waits (acquire), all leave together
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.tfull[a], use & 1u, abort_flag, kWaitNs))) break;
                tc::tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * kNV + quarter * kPassCols);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int v0 = t * kNV + 64 * h + kPassCols * quarter;
                    const int nvalid = min(16, p.V - v0);  // the same in the whole warp
                    float sv[16];
                    uint32_t uw[8];
                    __syncwarp();  // lanes that skipped the previous pass rejoin before the aligned load
                    tc::tmem_ld_32x32b_x16<0>(taddr + 64u * h, sv);
                    // this pass's base logits, then the buffer goes back to the U producer
                    // pass 2 g + h is in buffer (2 g + h) % kUBufs, filled for the
                    // ((2 g + h) / kUBufs)-th time
                    // (fused: the accumulator already holds U + B)
                    const int un = 2 * g + h, ub = un % kUBufs;
                    if constexpr (!kFused) {
                        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.ufull[ub], (uint32_t)((un / kUBufs) & 1),
                                                                   abort_flag, kWaitNs))) {
                            tc::tmem_ld_wait();
                            break;
                        }
                        const uint4 q0 = *reinterpret_cast<const uint4*>(sU + ub * kUBufBytes + u_off0);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(sU + ub * kUBufBytes + u_off1);
                        uw[0] = q0.x; uw[1] = q0.y; uw[2] = q0.z; uw[3] = q0.w;
                        uw[4] = q1.x; uw[5] = q1.y; uw[6] = q1.z; uw[7] = q1.w;
                    }
                    tc::tmem_ld_wait();
                    if (h == 1) {  // both halves are in registers: hand the accumulator back
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&bar.tempty[a]);
                    }
                    if constexpr (!kFused) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const uint32_t word = uw[c >> 1];
                            const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                            sv[c] = u + sv[c];  // the logit before the temperature
                        }
                        // the values are in registers: the async proxy may overwrite the buffer
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&bar.uempty[ub]);
                    }
                    if (row_ok && nvalid > 0) {
                        if (qrow) {  // scaled logits s = (U + B) / T
                            const float sc = sampling ? p.invT : 1.0f;
#pragma unroll
                            for (int c = 0; c < 16; c += 4)
                                if (c < nvalid)
                                    *reinterpret_cast<float4*>(qrow + v0 + c) =
                                        make_float4(sv[c] * sc, sv[c + 1] * sc, sv[c + 2] * sc, sv[c + 3] * sc);
                        }
                        if (p.greedy) {
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                if (c < nvalid && better(sv[c], v0 + c, part.score, part.idx)) {
                                    part.score = sv[c]; part.idx = v0 + c; part.s_at = sv[c];
                                }
                        } else {
                            // columns past the row end weigh 2^-inf = 0 and never pass the race test
                            if (nvalid < 16) {
#pragma unroll
                                for (int c = 0; c < 16; ++c)
                                    if (c >= nvalid) sv[c] = -INFINITY;
                            }
                            // Sampling draft in base 2: w = 2^(s * c2 - m2) with m2 a reference
                            // for the step's weights: the maximum of its first values, moved
                            // only when a pass's weights sum past 2^32 (an entry more than
                            // about 28 above it), so most passes need no maximum.  (max, sum)
                            // stays a valid log-sum-exp piece whatever the reference.
                            auto pass_max2 = [&]() {
                                float cm = sv[0];
#pragma unroll
                                for (int c = 1; c < 16; ++c) cm = fmaxf(cm, sv[c]);
                                return cm * c2;
                            };
                            // the tile's segment uniforms: pass h races with word 2 h and
                            // picks with word 2 h + 1 of counter 4 t + quarter
                            if (h == 0) {
                                uint4 x1[1] = {make_uint4((uint32_t)(4 * t + quarter), (uint32_t)pos, (uint32_t)rr, w3)};
                                philox4x32_10_xn<1>(x1, key0, key1);
                                seg_words = x1[0];
                            }
                            const uint32_t wu = h ? seg_words.z : seg_words.x;
                            const uint32_t wa = h ? seg_words.w : seg_words.y;
                            bool rec = false;  // this thread's record moved: publish it
                            if (part.m == -INFINITY) {
                                // the step's first values: their largest is the reference
                                const float cm = pass_max2();
                                if (cm > -INFINITY) part.m = cm;
                            }
                            if (part.m != -INFINITY) {  // else nothing finite yet
                                // rho bounds E / W of the row's winning segment in this thread's
                                // units (W = sum of 2^(s c2 - m)): this thread's record, or the
                                // best record G of the row's four quarters, E / W = 2^(m - G)
                                float gq;
                                {
                                    const unsigned long long raw =
                                        *reinterpret_cast<const volatile unsigned long long*>(&dsh.g[m][0]);
                                    const __half2 g01 = __halves2half2(__ushort_as_half((unsigned short)raw),
                                                                       __ushort_as_half((unsigned short)(raw >> 16)));
                                    const __half2 g23 = __halves2half2(__ushort_as_half((unsigned short)(raw >> 32)),
                                                                       __ushort_as_half((unsigned short)(raw >> 48)));
                                    const __half2 gm = __hmax2(g01, g23);
                                    gq = fmaxf(__low2float(gm), __high2float(gm));
                                }
                                rho = fminf(race_bound(bE, bw), ex2(part.m - gq) * kRaceSlack);
                                // the segment's weight, every entry of which goes into the normaliser
                                auto weigh = [&]() {
                                    const float nm = -part.m;
                                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                                    for (int c = 0; c < 16; ++c) acc[c & 3] += ex2(fmaf(sv[c], c2, nm));
                                    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
                                };
                                float ws = weigh();
                                if (!(ws <= 0x1p32f)) {
                                    // far above the reference (or a NaN): re-reference on this pass
                                    const float cm = pass_max2();
                                    if (cm > part.m) {
                                        const float sc = ex2(part.m - cm);
                                        part.sum *= sc;
                                        bw *= sc;
                                        part.m = cm;
                                        rho = fminf(race_bound(bE, bw), ex2(part.m - gq) * kRaceSlack);
                                        ws = weigh();
                                    }
                                }
                                part.sum += ws;
                                // the segment races with E = -ln u: it can replace the record only
                                // if 1 - u < W rho (E >= 1 - u), which needs no logarithm
                                if (one_plus_complement(wu) < fmaf(ws, rho, 1.0f)) {
                                    const float E = neg_log_uniform(wu);
                                    if (ws * bE > bw * E) {
                                        bw = ws; bE = E;
#pragma unroll
                                        for (int c = 0; c < 16; ++c) seg[c] = sv[c];
                                        seg_a = wa;
                                        seg_v0 = v0;
                                        rho = fminf(rho, race_bound(bE, bw));
                                        rec = true;
                                    }
                                }
                            }
                            if (rec)
                                *reinterpret_cast<volatile unsigned short*>(&dsh.g[m][quarter]) =
                                    __half_as_ushort(__float2half_rd(part.m + lg2(bw) - lg2(bE)));
                        }
                    }
                }
            }
            } else {
            // ---- residual: one race per request, over max(0, p - q) for a rejected
            // row and over p for a bonus draw (q = 0 there).  Thread = request row
            // m x 8 columns of each 32-column pass (pass h covers columns
            // 32 h + 8 quarter .. + 7 of a tile), four passes per tile.  The row's
            // target logits and base logits of the pass come from the staging
            // buffers (target rows:
            // 16-byte piece c of row m at m * 128 + (c ^ (m % 8)) * 16; base logits:
            // piece c of row m at m * 64 + (c ^ (m / 2 % 4)) * 16, so a warp's 32
            // rows read without bank conflicts).
            const int vq = 8 * quarter;
            const uint32_t t_off0 = (uint32_t)(m * 128 + (((2 * quarter) ^ (m & 7)) << 4));
            const uint32_t t_off1 = (uint32_t)(m * 128 + (((2 * quarter + 1) ^ (m & 7)) << 4));
            const uint32_t ru_off = (uint32_t)(m * 64 + ((quarter ^ ((m >> 1) & 3)) << 4));
            // pass n's 8 target logits (past the row end: zeros from the copy, read
            // as -inf: p = 0) and 8 base logits (bf16 pairs); the buffer then goes
            // back to the producer.  V % 8 == 0 and v % 8 == 0: a piece is wholly
            // inside or wholly past the row.  False when the wait gave up.
            auto take_piece = [&](int n, float (&tp)[8], uint32_t (&up)[4]) -> bool {
                const int b = n % kResBufs;
                if (!__all_sync(0xFFFFFFFFu,
                                tc::mbar_wait(&bar.sfull[b], (uint32_t)((n / kResBufs) & 1), abort_flag, kWaitNs)))
                    return false;
                const float4 f0 = *reinterpret_cast<const float4*>(sRT + b * kResTBytes + t_off0);
                const float4 f1 = *reinterpret_cast<const float4*>(sRT + b * kResTBytes + t_off1);
                const uint4 q = *reinterpret_cast<const uint4*>(sRU + b * kResUBytes + ru_off);
                tp[0] = f0.x; tp[1] = f0.y; tp[2] = f0.z; tp[3] = f0.w;
                tp[4] = f1.x; tp[5] = f1.y; tp[6] = f1.z; tp[7] = f1.w;
                up[0] = q.x; up[1] = q.y; up[2] = q.z; up[3] = q.w;
                // the values are in registers: the async proxy may overwrite the buffer
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bar.sempty[b]);
                return true;
            };
            // one pass: the accumulator's 8 columns at col, the piece at v0; last
            // hands the tile's accumulator back after reading it
            auto pass = [&](int v0, uint32_t col, bool last, int a, const float (&tp)[8],
                            const uint32_t (&up)[4]) {
                float sv[8];
                __syncwarp();  // lanes that skipped the previous pass rejoin before the aligned load
                tc::tmem_ld_32x32b_x8<0>(col, sv);
                tc::tmem_ld_wait();
                if (last) {
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bar.tempty[a]);
                }
                if (!(row_ok && v0 < p.V)) return;
                if (with_u) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t word = up[c >> 1];
                        const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                        sv[c] = (u + sv[c]) * c2;
                    }
                }
                uint4 x[2];
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    x[q] = make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)pos, (uint32_t)rr, w3);
                philox4x32_10_xn<2>(x, key0, key1);
                {
                    const float gq = fmaxf(fmaxf(g_own, g_glob),
                                           fmaxf(fmaxf(gsh[0], gsh[kM]), fmaxf(gsh[2 * kM], gsh[3 * kM])));
                    rho = fminf(race_bound(bE, bw), ex2(-gq) * kRaceSlack);
                }
                float wv[8];
                uint32_t cand = 0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float pv = ex2(fmaf(tp[c], c2, -rinfo.lse2_p));
                    const float wgt = with_u ? pv - ex2(sv[c] - rinfo.q_lse2) : pv;
                    wv[c] = wgt;
                    cand |= (wgt > 0.0f && one_plus_complement(word_of(x[c >> 2], c & 3)) < fmaf(wgt, rho, 1.0f))
                                ? (1u << c)
                                : 0u;
                }
                if (cand) {
                    // this lane's candidates one at a time, lowest column first
                    bool rec = false;
                    const uint32_t words[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
                    do {
                        const int c = __ffs(cand) - 1;
                        cand &= cand - 1u;
                        const float w = pick<8>(wv, c);
                        const float E = neg_log_uniform(pick<8>(words, c));
                        if (w * bE > bw * E) {
                            bw = w; bE = E; part.idx = v0 + c;
                            rho = fminf(rho, race_bound(bE, bw));
                            rec = true;
                        }
                    } while (cand);
                    if (rec) {
                        g_own = lg2(bw) - lg2(bE);
                        gsh[quarter * kM] = g_own;
                    }
                }
            };
            for (int i = 0; staged && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                const int a = i & 1;  // one step: the launch's tile index is i
                const uint32_t use = (uint32_t)(i >> 1);
                if (share) {
                    if (i > 0) g_glob = key_log2_ratio(gkey);
                    gkey = *reinterpret_cast<volatile unsigned long long*>(my_key);
                }
                // warp-uniform wait: every lane waits (acquire), all leave together
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.tfull[a], use & 1u, abort_flag, kWaitNs))) break;
                tc::tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * kNV + vq);
                const int vt = t * kNV + vq;
#pragma unroll 1
                for (int h = 0; h < 4; ++h) {
                    float tp[8];
                    uint32_t up[4];
                    const int n = 4 * i + h;
                    if (n + kResAhead < n_res && !stage_issue(n + kResAhead)) { staged = false; break; }
                    if (!take_piece(n, tp, up)) { staged = false; break; }
                    pass(vt + kResCols * h, taddr + (uint32_t)(kResCols * h), h == 3, a, tp, up);
                }
                if (!staged) break;
                // this thread's record, if it beats the request's best seen so far, for the
                // other CTAs racing over it (few threads qualify after the first tiles:
                // same-address atomics serialise)
                if (share && g_own > fmaxf(g_pub, g_glob)) {
                    atomicMax(my_key, winner_key(logf(bw) - logf(bE), part.idx));
                    g_pub = g_own;
                }
            }
            // staging copies still in flight (after an abort) land before the CTA exits
            cp_async_wait_all();
            }
            // scores of the winners in log form, for merging across threads and CTAs
            if (kRes) {
                part.score = part.idx != INT_MAX ? logf(bw) - logf(bE) : -INFINITY;
            } else if (!p.greedy) {
                if (bw > 0.0f) {
                    // the entry of the record segment: the first whose running sum of
                    // weights passes a times the segment's total (weights relative to
                    // the segment's own largest value, so none underflows)
                    float mx = seg[0];
#pragma unroll
                    for (int c = 1; c < 16; ++c) mx = fmaxf(mx, seg[c]);
                    const float nm = -mx * c2;
                    float wt[16];
                    float tot = 0.0f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        wt[c] = ex2(fmaf(seg[c], c2, nm));
                        tot += wt[c];
                    }
                    const float target = uniform_from_bits(seg_a) * tot;
                    // upward: the first c whose running sum passes the target; failing
                    // that (rounding), the last entry with weight
                    int pick_c = -1, last_c = 0;
                    float run = 0.0f, s_pick = seg[0];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        run += wt[c];
                        if (wt[c] > 0.0f && pick_c < 0) { last_c = c; }
                        if (pick_c < 0 && run > target) { pick_c = c; s_pick = seg[c]; }
                    }
                    if (pick_c < 0) {
                        pick_c = last_c;
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            if (c == last_c) s_pick = seg[c];
                    }
                    part.idx = seg_v0 + pick_c;
                    part.s_at = s_pick * c2;
                    // the segment's race value log W - log E in natural units
                    part.score = fmaf(part.m + lg2(bw), kLn2F, -logf(bE));
                }
                // back to natural units: the max and the winner's logit
                part.m *= kLn2F;
                part.s_at *= kLn2F;
            }

            // ---- the CTA's result of the step: the row's four quarters merged by
            // quarter 0, which publishes the winner key and (draft) the normaliser piece
            if (quarter != 0) scratch[(quarter - 1) * kM + m] = part;
            epi_sync();
            if (quarter == 0 && row_ok && !*abort_flag) {
#pragma unroll
                for (int q = 0; q < 3; ++q) merge_any<kRes>(part, scratch[q * kM + m]);
                if (kRes) {
                    if (part.idx != INT_MAX) atomicMax(p.keys + rr, winner_key(part.score, part.idx));
                } else {
                    const size_t slot = (size_t)k * p.R + rr;
                    if (!p.greedy)
                        p.parts[slot * p.P + cidx] = make_float4(part.m, part.sum, part.s_at, __int_as_float(part.idx));
                    if (part.idx != INT_MAX && IN_BOUNDS(part.idx >= 0 && part.idx < p.V, p.dev_status))
                        atomicMax(p.keys + slot, winner_key(part.score, part.idx));
                }
            }
            if (k + 1 < n_steps) {
                // ---- every CTA's keys of step k before any CTA reads them (the scratch
                // is free again after this too)
                epi_sync();
                if (e == 0) {
                    bool ok = !*abort_flag;
                    if (ok)
                        ok = step_barrier(p.step_done + k, reinterpret_cast<int*>(p.step_done + p.gamma),
                                          gridDim.x + p.phantom, p.wait_ns);
                    else atomicExch(reinterpret_cast<int*>(p.step_done + p.gamma), 1);
                    if (!ok) *abort_flag = 1;  // the control warps stop too
                    bar.step_ok = ok ? 1 : 0;
                }
                epi_sync();
                if (!bar.step_ok) break;
            }
        }
        if constexpr (!kRes) {
            // ---- after the last position: every CTA's keys and pieces are
            // published (the last counter) before any CTA reads them, then each
            // epilogue warp of the grid finalizes (position, request) pairs: the
            // token from the winner key, the log-normaliser from the CTAs' (max,
            // sum) pieces, q(y) from the piece of the CTA that held the winner.  A
            // request without a key had an unusable anchor or predecessor (or no
            // finite logit): its token is -1 and its q values NaN.
            epi_sync();
            if (e == 0) {
                int* abort_word = reinterpret_cast<int*>(p.step_done + p.gamma);
                bool ok = !*abort_flag;
                if (ok) ok = step_barrier(p.step_done + (p.gamma - 1), abort_word, gridDim.x + p.phantom, p.wait_ns);
                else atomicExch(abort_word, 1);
                if (!ok) *abort_flag = 1;
                bar.step_ok = ok ? 1 : 0;
            }
            epi_sync();
            if (bar.step_ok) {
                const int n_pairs = p.gamma * p.R;
                const int gw_stride = (int)gridDim.x * kEpiWarps;
                for (int pr = (int)blockIdx.x * kEpiWarps + ew; pr < n_pairs; pr += gw_stride) {
                    const int k = pr / p.R, r = pr - k * p.R;
                    const size_t slot = (size_t)k * p.R + r;
                    const size_t rk = (size_t)r * p.gamma + k;
                    const unsigned long long key = __ldcg(p.keys + slot);
                    if (key == 0) {
                        if (lane == 0) {
                            p.y[rk] = -1;
                            if (!p.greedy) {
                                if (p.q_lse) p.q_lse[rk] = NAN;
                                if (p.q_tok) p.q_tok[rk] = NAN;
                            }
                            report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
                        }
                        continue;
                    }
                    const int idx = key_index(key);
                    if (!IN_BOUNDS(idx >= 0 && idx < p.V, p.dev_status)) {
                        if (lane == 0) p.y[rk] = -1;
                        continue;
                    }
                    if (p.greedy) {
                        if (lane == 0) p.y[rk] = idx;
                        continue;
                    }
                    float fm = -INFINITY, fs = 0.0f, sat = -INFINITY;
                    for (int j = lane; j < p.P; j += 32) {
                        const float4 q = __ldcg(p.parts + slot * p.P + j);
                        lse_merge(fm, fs, q.x, q.y);
                        if (__float_as_int(q.w) == idx) sat = q.z;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float m2 = shfl_xor(fm, o), s2 = shfl_xor(fs, o);
                        lse_merge(fm, fs, m2, s2);
                        sat = fmaxf(sat, shfl_xor(sat, o));
                    }
                    if (lane == 0) {
                        const float lse = fm + logf(fs);
                        p.y[rk] = idx;
                        if (p.q_lse) p.q_lse[rk] = lse;
                        if (p.q_tok) p.q_tok[rk] = expf(sat - lse);
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (*abort_flag && threadIdx.x == 0) report(p.dev_status, DSPARK_ERR_TIMEOUT);
    if constexpr (kRes) residual_tokens_if_last(p, smem, bar);
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    }
    return fn;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: winner keys (residual: and after them the count of CTAs done),
// (draft) the step counters and the abort word of the launch's grid barrier,
// zeroed with the keys, then (draft) the per-CTA normaliser pieces or
// (residual) the per-request rows.
struct TcLayout {
    size_t keys, n_keys, step_done, zero_bytes, parts, rows, total;
};
TcLayout tc_layout(int R, int gamma, bool residual) {
    TcLayout L;
    size_t off = 0;
    L.n_keys = residual ? (size_t)R + 1 : (size_t)gamma * R;  // residual: + the count of CTAs done
    L.keys = off; off += sizeof(unsigned long long) * L.n_keys;
    L.step_done = off; off += residual ? 0 : sizeof(unsigned) * ((size_t)gamma + 1);
    L.zero_bytes = off;
    off = up256(off);
    L.parts = off; off += residual ? 0 : up256(sizeof(float4) * (size_t)gamma * R * kMaxP);
    L.rows = off; off += residual ? up256(sizeof(ResRow) * (size_t)R) : 0;
    L.total = off;
    return L;
}

bool encode_2d_bf16(EncodeTiled enc, CUtensorMap* m, const void* base, int inner, int outer, int box_outer) {
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t box[2] = {kKB, (cuuint32_t)box_outer};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared launch setup of both modes: device limits, stage count, tensor maps,
// the common parameter block.  Returns DSPARK_OK or an error status.
// d > 0: the fused draft, with h [R, gamma, d] in place of U and the lm_head
// W_lm [V, d] (tm_wlm; otherwise tm_wlm is a copy of tm_w2, unused).
int prepare(EncodeTiled enc, const void* U, const void* W1, const void* W2, int R, int gamma, int V, int rank,
            bool residual, const void* W_lm, int d, TcParams& p, CUtensorMap& tm_w2, CUtensorMap& tm_u,
            CUtensorMap& tm_wlm, int& grid, size_t& smem, int& n_sm) {
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int nkb = rank / kKB;
    // A lives in tensor memory; shared memory holds the residual's staging
    // buffers, or the draft's quarter exchange and U pass buffers, then the ring
    const bool fused = d > 0;
    const size_t fixed =
        1024 + sizeof(Bars) +
        (residual ? kShareBytes + (size_t)kResBufs * (kResTBytes + kResUBytes)
                  : sizeof(DraftShared) + (size_t)kExchBytes + (fused ? 0 : (size_t)kUBufs * kUBufBytes));
    // the residual's end-of-step exchange reuses the drained W2 ring (at least two stages)
    static_assert(2 * kTileBytes >= 3 * kM * sizeof(TcPartial), "exchange larger than two ring stages");
    const size_t stage = fused ? 2 * (size_t)kTileBytes : (size_t)kTileBytes;
    if ((size_t)max_smem < fixed + 2 * stage) return DSPARK_ERR_UNSUPPORTED;
    const int n_stages = (int)std::min<size_t>(kMaxStages, ((size_t)max_smem - fixed) / stage);
    smem = fixed + (size_t)n_stages * stage;

    if (!encode_2d_bf16(enc, &tm_w2, W2, rank, V, kNV)) return DSPARK_ERR_CUDA;
    tm_wlm = tm_w2;
    if (fused && !encode_2d_bf16(enc, &tm_wlm, W_lm, d, V, kNV)) return DSPARK_ERR_CUDA;
    if (!residual) {
        // U [R, gamma, V], or the fused draft's h [R, gamma, d]: boxes of 64 x 1 x 128
        const int inner = fused ? d : V;
        const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)gamma, (cuuint64_t)R};
        const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)gamma * inner * 2};
        const cuuint32_t box[3] = {kKB, 1, kM};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tm_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_CUDA;
    } else {
        tm_u = tm_w2;  // unused by the residual
    }
    p = TcParams();
    p.U = static_cast<const uint16_t*>(U);
    p.W1 = static_cast<const uint16_t*>(W1);
    p.w1_wide = (reinterpret_cast<uintptr_t>(W1) & 31u) == 0;
    p.R = R;
    p.gamma = gamma;
    p.V = V;
    p.rank = rank;
    p.nb = (R + kM - 1) / kM;
    p.n_tiles = (V + kNV - 1) / kNV;
    p.P = std::max(1, std::min(std::min(n_sm / p.nb, p.n_tiles), kMaxP));
    p.n_stages = n_stages;
    p.nkb = nkb;
    p.dkb = fused ? d / kKB : 0;
    grid = p.P * p.nb;
    return DSPARK_OK;
}

}  // namespace

bool draft_tc_fits(int R) {
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    return (R + kM - 1) / kM <= n_sm;
}

bool draft_tc_supported(int u_dtype, int w_dtype, int R, int V, int rank) {
    return u_dtype == DSPARK_BF16 && w_dtype == DSPARK_BF16 && R >= 1 && rank % kKB == 0 && rank >= kKB &&
           rank <= 512 && V % 8 == 0 && V >= 8;
}

size_t draft_tc_workspace(int R, int gamma, int /*rank*/) { return tc_layout(R, gamma, false).total; }

size_t residual_tc_workspace(int R, int /*rank*/) { return tc_layout(R, 0, true).total; }

ResRow* residual_tc_rows(void* ws, int R) {
    return reinterpret_cast<ResRow*>(static_cast<unsigned char*>(ws) + tc_layout(R, 0, true).rows);
}

unsigned long long* residual_tc_keys(void* ws, int R) {
    return reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(ws) + tc_layout(R, 0, true).keys);
}

int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    if (a.q_logits && (reinterpret_cast<uintptr_t>(a.q_logits) & 15)) return DSPARK_ERR_UNSUPPORTED;
    const TcLayout L = tc_layout(a.R, a.gamma, false);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_wlm;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const bool fused = a.d > 0;
    const int st = prepare(enc, fused ? a.h : a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, false, a.W_lm, a.d, p,
                           tm_w2, tm_u, tm_wlm, grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    p.keys = reinterpret_cast<unsigned long long*>(w + L.keys);
    p.step_done = reinterpret_cast<unsigned*>(w + L.step_done);
    p.parts = reinterpret_cast<float4*>(w + L.parts);
    p.anchor = a.anchor;
    p.seeds = a.seeds;
    p.q_logits = a.q_logits;
    p.y = a.y;
    p.q_lse = a.q_lse;
    p.q_tok = a.q_tok;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = a.greedy;
    p.wait_ns = grid_wait_limit_ns();
    p.phantom = (fault_injection_mask() & DSPARK_INJECT_DRAFT_BARRIER) ? 1u : 0u;
    auto kern = fused ? markov_tc_kernel<false, true> : markov_tc_kernel<false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    // keys, step counters and abort word in one piece
    if (cudaMemsetAsync(w, 0, L.zero_bytes, stream) != cudaSuccess) return DSPARK_ERR_CUDA;
    // All gamma steps in one launch whose CTAs wait for one another between
    // steps: a cooperative launch, so that every CTA is resident (one per SM,
    // grid <= SM count) or the launch fails.
    cudaLaunchAttribute coop[1];
    coop[0].id = cudaLaunchAttributeCooperative;
    coop[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = coop;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tm_w2, tm_u, tm_wlm, p) != cudaSuccess) return DSPARK_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int launch_residual_tc(const ResidualTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    const TcLayout L = tc_layout(a.R, a.gamma, true);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_wlm;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st = prepare(enc, a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, true, nullptr, 0, p, tm_w2, tm_u, tm_wlm,
                           grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    ResRow* rows = reinterpret_cast<ResRow*>(w + L.rows);
    p.keys = reinterpret_cast<unsigned long long*>(w + L.keys);  // zeroed by the verify prologue
    p.seeds = a.seeds;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = 0;
    p.target = a.target;
    p.rows = rows;
    p.out_tokens = a.out_tokens;
    p.wait_ns = kWaitNs;  // no grid barrier in the residual launch
    p.phantom = 0;
    if (cudaFuncSetAttribute(markov_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    markov_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tm_w2, tm_u, tm_wlm, p);
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark

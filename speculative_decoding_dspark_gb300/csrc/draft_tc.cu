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
//   draft     one launch per position k: logits of every request, Gumbel-max
//             sample and the pieces of its log-normaliser and q(y);
//   residual  one launch per verify: for every request the drafter's logits of
//             its rejected row are recomputed here (the residual needs q on the
//             whole vocabulary, and recomputing one row per request costs one
//             pass over W2 instead of keeping every drafted row in memory),
//             then the extra token is drawn from max(0, p - q), or from p after
//             full acceptance.
//
// Persistent, one CTA per SM, 19 warps:
//   A (M = 128 requests x K = rank) = rows W1[prev], gathered once per launch
//     into a workspace matrix H by a small kernel (spread over many SMs: the
//     rows are scattered over W1's pages), loaded by TMA into 128-byte-swizzled
//     shared memory and resident for the launch;
//   B (N = 128 vocabulary rows x K = rank) = W2 tiles streamed by TMA through a
//     ring of 16 KB stages; the next tile's boxes are prefetched into L2 one
//     tile ahead so the ring only has to cover L2 latency;
//   D = A . B^T in fp32 tensor memory, two 128-column buffers so the epilogue
//     of one vocabulary tile overlaps the MMAs of the next;
//   U_k (draft) = the tile's base logits, by TMA into two 16 KB pass buffers
//     (128 requests x 64 columns, 128-byte-swizzled) one pass ahead of the
//     epilogue, which adds them to the accumulator;
//   epilogue (16 warps; thread = one request x 32 vocabulary columns of a
//     tile, in two 16-column passes, pass h over columns 64 h .. 64 h + 63 of
//     the tile across the four warps of a lane quadrant): Gumbel-max draws
//     use the exponential-race form: with
//     weight w > 0 and E = -log(u), the largest log(w) + Gumbel(u) is the
//     largest w / E, so a candidate replaces the best when
//     w * E_best > w_best * E.  Since E >= 1 - u, an entry with
//     1 - u >= w * E_best / w_best cannot win; that test needs no logarithm
//     (1 - u comes exactly from the random bits), and only the entries that
//     pass it take the log (a short series in 1 - u near u = 1, the
//     special-function log2 elsewhere; relative error about 2e-6) and the
//     comparison.
//
// Cross-CTA results need no merging pass: every CTA folds its winner into one
// 64-bit key per request and step with atomicMax (order-preserving bits of
// the score above the inverted index, so ties go to the lower index), and
// stores its (max, sum of exp, winner logit) piece of the normaliser.  The
// next draft step decodes its A rows' tokens from the keys (it is launched
// as a programmatic dependent and waits for the previous step before reading
// them, while its producer already streams W2), and one finalize kernel after
// the last step turns keys and pieces into tokens, q_lse and q(y).  The chain
// gather -> step -> gather -> ... -> finalize is launched with programmatic
// stream serialization: each launch starts as the previous one retires, its
// producers pull its first W2 and U tiles into L2, and only reading H / the
// keys waits for the previous launch to complete.
//
// Warp roles: warp 0 = W2/A TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warp 2 = U TMA producer (draft), warps 3-18 = epilogue.  Every mbarrier wait is bounded (2 s);
// a timeout aborts the CTA cleanly and reports DSPARK_ERR_TIMEOUT.
#include <cuda.h>

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
constexpr int kMaxStages = 8;
constexpr int kMaxP = 256;                    // CTAs per request block (pieces per request)
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
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

// Per-request description of the residual launch.
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

struct TcParams {
    const uint16_t* U;
    const uint16_t* W1;
    unsigned long long* keys;  // draft [gamma][R]; residual [R]
    const int32_t* toks;       // draft [R]: the A rows' tokens (-2: no usable predecessor)
    float4* parts;             // draft [gamma][R][P]: (max, sum, winner logit, winner) per CTA
    const uint64_t* seeds;
    int32_t* dev_status;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank, k;
    int nb, P, n_tiles, n_stages, nkb;
    const int32_t* anchor;
    float* q_logits;
    const float* target;
    const ResRow* rows;
};

struct Bars {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t tfull[2], tempty[2];
    uint64_t ufull[2], uempty[2];
    uint64_t afull, mma_done;
    uint32_t tmem_slot;
    int abort_flag;
    // per request row and epilogue quarter: the best race record so far as
    // log2(w / E) in absolute units (-inf: none), read by the row's other quarters
    float g_share[4][kM];
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

__device__ __forceinline__ uint32_t word_of(const uint4& x, int j) {
    return j == 0 ? x.x : (j == 1 ? x.y : (j == 2 ? x.z : x.w));
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on to
// complete (and their writes to be visible); allow dependents to be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Copies W1[t] (zeros for t < 0) into row r of H: one warp, 16-byte pieces.
__device__ __forceinline__ void copy_w1_row(const uint16_t* W1, int t, int rank, uint16_t* H, int r, int lane) {
    const int cpr = rank >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(W1 + (size_t)(t < 0 ? 0 : t) * rank);
    uint4* dst = reinterpret_cast<uint4*>(H + (size_t)r * rank);
    for (int c = lane; c < cpr; c += 32) dst[c] = t >= 0 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
}

// The A rows of draft step k, one small CTA per request (the rows lie on
// scattered pages of W1; one row per SM keeps the address translations of the
// gather in parallel): the predecessor token (the anchor at k = 0, else the
// winner of step k - 1 decoded from its key; -1 no anchor, -2 unusable: the
// step then computes nothing for the request) and its W1 row.
constexpr int kGatherThreads = 64;
__global__ void __launch_bounds__(kGatherThreads) gather_a_rows_kernel(const uint16_t* W1, const int32_t* anchor,
                                                                       const unsigned long long* prev_keys, int k,
                                                                       int R, int V, int rank, uint16_t* H,
                                                                       int32_t* toks) {
    griddep_launch_dependents();
    griddep_wait();  // the previous step's keys
    const int r = blockIdx.x;
    int t;
    if (k == 0) {
        const int a = anchor[r];
        t = a >= V ? -2 : (a < 0 ? -1 : a);
    } else {
        const unsigned long long key = prev_keys[r];
        t = key ? key_index(key) : -2;
    }
    if (threadIdx.x == 0) toks[r] = t;
    const int cpr = rank >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(W1 + (size_t)(t < 0 ? 0 : t) * rank);
    uint4* dst = reinterpret_cast<uint4*>(H + (size_t)r * rank);
    for (int c = threadIdx.x; c < cpr; c += kGatherThreads) dst[c] = t >= 0 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
}

// Per request after the verify decisions: what the residual launch draws, and
// its A row W1[prev] of the rejected position (zeros for a bonus draw).  One
// warp per request.
__global__ void __launch_bounds__(256) residual_prep_kernel(ResidualTcArgs a, ResRow* rows, uint16_t* H) {
    const int r = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= a.R) return;
    const VerifyJob job = a.jobs[r];
    const int mode = a.valid[r] ? job.mode : 0;
    int prev = -1;
    if (mode == 1) {
        prev = job.pos == 0 ? a.anchor[r] : a.y[(size_t)r * a.gamma + job.pos - 1];
        if (prev >= a.V || prev < 0) prev = -1;
    }
    ResRow w;
    w.mode = mode;
    w.pos = job.pos;
    w.trow = job.row;
    w.w3 = ctr_word3(a.cycle, mode == 1 ? kResidualGumbel : kBonusGumbel);
    w.lse2_p = job.lse * kLog2eF;
    w.q_lse2 = mode == 1 ? a.q_lse[(size_t)r * a.gamma + job.pos] * kLog2eF : 0.0f;
    w.prev = prev;
    w.pad = 0.0f;
    if (lane == 0) rows[r] = w;
    copy_w1_row(static_cast<const uint16_t*>(a.W1), prev, a.rank, H, r, lane);
}

template <bool kRes>
__global__ void __launch_bounds__(kThreads, 1)
markov_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
                 const __grid_constant__ CUtensorMap tm_h, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sU = sA + p.nkb * kTileBytes;          // draft: two pass buffers of base logits
    uint8_t* sB = sU + (kRes ? 0 : 2 * kUBufBytes);
    Bars& bar = *reinterpret_cast<Bars*>(sB + p.n_stages * kTileBytes);
    volatile int* abort_flag = &bar.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = blockIdx.x % p.nb;
    const int cidx = blockIdx.x / p.nb;
    const int row0 = blk * kM;
    const int S = p.n_stages;

    for (int e = threadIdx.x; e < 4 * kM; e += kThreads) (&bar.g_share[0][0])[e] = -INFINITY;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { tc::mbar_init(&bar.full[s], 1); tc::mbar_init(&bar.empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar.tfull[a], 1); tc::mbar_init(&bar.tempty[a], kEpiWarps); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar.ufull[a], 1); tc::mbar_init(&bar.uempty[a], kEpiWarps); }
        tc::mbar_init(&bar.afull, 1);
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
        tc::prefetch_tmap(&tm_h);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    // The next launch may be scheduled as SMs free up; it waits (griddepcontrol)
    // before it reads anything this one writes.
    griddep_launch_dependents();
    const uint32_t tmem_base = bar.tmem_slot;
    const int n_local = cidx < p.n_tiles ? (p.n_tiles - 1 - cidx) / p.P + 1 : 0;

    // this thread's running partial (epilogue threads)
    TcPartial part = identity_partial<kRes>();
    bool row_ok = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // W2 and U are inputs no launch of this library writes: the first tiles
        // are requested into L2 before waiting for the previous launch, which
        // wrote H; A is loaded first, then the W2 ring.
        if (lane == 0) {
            for (int i = 0; i < 2 && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                for (int q = 0; q < p.nkb; ++q) tma_prefetch_l2_2d(&tm_w2, q * kKB, t * kNV);
                if (!kRes) {
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV, p.k, row0);
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV + kKB, p.k, row0);
                }
            }
            const int n_loads = n_local * p.nkb;  // W2 stage loads, tile-major
            int issued = 0;
            bool ok = true;
            // the stage of load l is l % S, used for the (l / S)-th time
            auto issue = [&](int l) {
                const int s = l % S, i = l / p.nkb, kb = l - i * p.nkb;
                const int t = cidx + i * p.P;
                tc::mbar_arrive_expect_tx(&bar.full[s], kTileBytes);
                tc::tma_load_2d(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV);
                // once a tile's first ring of loads is out, pull the next tile into L2
                if (kb == min(S, p.nkb) - 1 && i + 1 < n_local) {
                    const int tn = t + p.P;
                    for (int q = 0; q < p.nkb; ++q) tma_prefetch_l2_2d(&tm_w2, q * kKB, tn * kNV);
                    if (!kRes) {
                        tc::tma_prefetch_l2_3d(&tm_u, tn * kNV, p.k, row0);
                        tc::tma_prefetch_l2_3d(&tm_u, tn * kNV + kKB, p.k, row0);
                    }
                }
            };
            griddep_wait();
            // A: the block's H rows, resident for the launch
            tc::mbar_arrive_expect_tx(&bar.afull, (uint32_t)(p.nkb * kTileBytes));
            for (int kb = 0; kb < p.nkb; ++kb) tc::tma_load_2d(sA + kb * kTileBytes, &tm_h, &bar.afull, kb * kKB, row0);
            for (; issued < n_loads; ++issued) {
                const int s = issued % S;
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                if (!tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs)) { ok = false; break; }
                issue(issued);
            }
            // the copies this thread issued must land before the CTA exits
            int dummy = 0;
            volatile int* no_abort = &dummy;
            tc::mbar_wait(&bar.afull, 0, no_abort, kWaitNs);
            if (!ok) {
                for (int l = max(0, issued - S); l < issued; ++l)
                    tc::mbar_wait(&bar.full[l % S], (uint32_t)((l / S) & 1), no_abort, kWaitNs);
            }
        }
        __syncwarp();  // the warp reconverges before the CTA-wide barrier below
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kM, kNV);
            bool ok = tc::mbar_wait(&bar.afull, 0, abort_flag, kWaitNs);
            tc::tc_fence_after();
            int s = 0;
            uint32_t ph = 0;
            const uint32_t a_base = tc::smem_u32(sA), b_base = tc::smem_u32(sB);
            for (int i = 0; ok && i < n_local; ++i) {
                const int a = i & 1;
                const uint32_t use = (uint32_t)(i >> 1);
                if (!tc::mbar_wait(&bar.tempty[a], (use & 1u) ^ 1u, abort_flag, kWaitNs)) { ok = false; break; }
                tc::tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kNV);
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!tc::mbar_wait(&bar.full[s], ph, abort_flag, kWaitNs)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t aa = a_base + (uint32_t)(kb * kTileBytes);
                    const uint32_t bb = b_base + (uint32_t)(s * kTileBytes);
#pragma unroll
                    for (int j = 0; j < kKB / 16; ++j)
                        tc::umma_bf16(d, tc::smem_desc_sw128(aa + 32u * j), tc::smem_desc_sw128(bb + 32u * j), idesc,
                                      (kb | j) != 0);
                    tc::umma_commit(&bar.empty[s]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc::umma_commit(&bar.tfull[a]);
            }
            // every MMA issued has completed before anyone frees tensor memory
            tc::umma_commit(&bar.mma_done);
            int dummy = 0;
            volatile int* no_abort = &dummy;
            tc::mbar_wait(&bar.mma_done, 0, no_abort, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ U producer
        // Draft: the base logits U_k of pass n (tile n / 2, columns 64 (n % 2) ..
        // + 63 of the tile, all 128 requests) into pass buffer n % 2, one pass ahead
        // of the epilogue; U is an input, so no wait on the previous launch.
        if (!kRes && lane == 0) {
            const int n_pass = 2 * n_local;
            int n = 0;
            for (; n < n_pass; ++n) {
                const int b = n & 1;
                const uint32_t use = (uint32_t)(n >> 1);
                if (!tc::mbar_wait(&bar.uempty[b], (use & 1u) ^ 1u, abort_flag, kWaitNs)) break;
                tc::mbar_arrive_expect_tx(&bar.ufull[b], (uint32_t)kUBufBytes);
                tc::tma_load_3d(sU + b * kUBufBytes, &tm_u, &bar.ufull[b], (cidx + (n >> 1) * p.P) * kNV + 64 * b, p.k,
                                row0);
            }
            // the copies this thread issued must land before the CTA exits
            int dummy = 0;
            volatile int* no_abort = &dummy;
            for (int l = max(0, n - 2); l < n; ++l)
                tc::mbar_wait(&bar.ufull[l & 1], (uint32_t)((l >> 1) & 1), no_abort, kWaitNs);
        }
        __syncwarp();
    } else {
        // the A rows' tokens (draft) were written by the previous launch
        griddep_wait();
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kCtlWarps;   // 0..15
        const int quad = warp & 3;         // TMEM lane quadrant this warp may read
        const int quarter = ew >> 2;       // pass h covers columns 64 h + 16 quarter .. + 15 of a tile
        const int m = quad * 32 + lane;
        const int rr = row0 + m;
        if (kRes) row_ok = rr < p.R && p.rows[rr].mode != 0;
        else row_ok = rr < p.R && p.toks[rr] != -2;
        ResRow rinfo;
        rinfo.mode = 0; rinfo.pos = 0; rinfo.trow = 0; rinfo.w3 = 0; rinfo.lse2_p = 0.0f; rinfo.q_lse2 = 0.0f;
        if (kRes && row_ok) rinfo = p.rows[rr];
        const bool sampling = kRes || !p.greedy;
        const uint64_t seed = (sampling && row_ok) ? p.seeds[rr] : 0ull;
        const uint32_t key0 = (uint32_t)(seed & 0xFFFFFFFFu), key1 = (uint32_t)(seed >> 32);
        const uint32_t w3 = kRes ? rinfo.w3 : ctr_word3(p.cycle, kDraftGumbel);
        const int pos = kRes ? rinfo.pos : p.k;
        const bool with_u = !kRes || rinfo.mode == 1;
        const size_t rk = (size_t)rr * p.gamma + pos;
        const uint16_t* urow = p.U + rk * p.V;
        const float* trow = kRes ? p.target + (size_t)rinfo.trow * p.V : nullptr;
        float* qrow = (!kRes && p.q_logits && row_ok) ? p.q_logits + rk * p.V : nullptr;
        // logits are scaled to base 2 when sampling: s2 = s * log2(e) / T
        const float c2 = sampling ? p.invT * kLog2eF : 1.0f;
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
        float g_own = -INFINITY, g_pub = -INFINITY, g_glob = -INFINITY;
        unsigned long long gkey = 0;
        const bool share = kRes && row_ok;
        unsigned long long* my_key = kRes ? p.keys + rr : p.keys + (size_t)p.k * p.R + rr;
        volatile float* gsh = &bar.g_share[0][m];  // the row's four quarter records, written by other warps
        // residual: the 16 base logits (bf16 pairs) of the request's rejected row at v
        auto load_u = [&](int v, uint32_t(&dst)[8]) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 q = (row_ok && v + 8 * j < p.V) ? __ldg(reinterpret_cast<const uint4*>(urow + v) + j)
                                                             : make_uint4(0u, 0u, 0u, 0u);
                dst[4 * j + 0] = q.x; dst[4 * j + 1] = q.y; dst[4 * j + 2] = q.z; dst[4 * j + 3] = q.w;
            }
        };
        // draft: this thread's 32 bytes of a pass buffer (row m, 16-byte chunks
        // 2 quarter and 2 quarter + 1 of the 128-byte-swizzled row)
        const uint32_t u_off0 = (uint32_t)(m * 128 + (((2 * quarter) ^ (m & 7)) << 4));
        const uint32_t u_off1 = (uint32_t)(m * 128 + (((2 * quarter + 1) ^ (m & 7)) << 4));
        for (int i = 0; i < n_local; ++i) {
            const int t = cidx + i * p.P;
            const int a = i & 1;
            const uint32_t use = (uint32_t)(i >> 1);
            if (kRes && row_ok) {
                // residual rows differ per request: pull this thread's pieces of the
                // next tile (of this one too, at the start) into L2
                for (int tt = (i == 0 ? t : t + p.P); tt <= t + p.P && tt < p.n_tiles; tt += p.P) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int v = tt * kNV + 64 * h + kPassCols * quarter;
                        if (v < p.V) {
                            prefetch_l2(trow + v);
                            if (with_u) prefetch_l2(urow + v);
                        }
                    }
                }
            }
            if (share) {
                if (i > 0) g_glob = key_log2_ratio(gkey);
                gkey = *reinterpret_cast<volatile unsigned long long*>(my_key);
            }
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
                float tv[16];
                if constexpr (kRes) {
                    // residual: target logits (past the row end -inf: p = 0) and, for a
                    // rejected row, the drafter's base logits; requested before the
                    // accumulator is read
                    if (row_ok && nvalid > 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 f = 4 * j < nvalid ? __ldg(reinterpret_cast<const float4*>(trow + v0) + j)
                                                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                            tv[4 * j + 0] = f.x; tv[4 * j + 1] = f.y; tv[4 * j + 2] = f.z; tv[4 * j + 3] = f.w;
                        }
                        if (with_u) load_u(v0, uw);
                    }
                }
                __syncwarp();  // lanes that skipped the previous pass rejoin before the aligned load
                tc::tmem_ld_32x32b_x16<0>(taddr + 64u * h, sv);
                if (!kRes) {
                    // this pass's base logits, then the buffer goes back to the U producer
                    // pass buffer h is filled once per tile: its phase parity is i & 1
                    if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.ufull[h], (uint32_t)(i & 1), abort_flag, kWaitNs))) {
                        tc::tmem_ld_wait();
                        break;
                    }
                    const uint4 q0 = *reinterpret_cast<const uint4*>(sU + h * kUBufBytes + u_off0);
                    const uint4 q1 = *reinterpret_cast<const uint4*>(sU + h * kUBufBytes + u_off1);
                    uw[0] = q0.x; uw[1] = q0.y; uw[2] = q0.z; uw[3] = q0.w;
                    uw[4] = q1.x; uw[5] = q1.y; uw[6] = q1.z; uw[7] = q1.w;
                }
                tc::tmem_ld_wait();
                if (h == 1) {  // both halves are in registers: hand the accumulator back
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bar.tempty[a]);
                }
                if (!kRes) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint32_t word = uw[c >> 1];
                        const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                        sv[c] = (u + sv[c]) * c2;
                    }
                    // the values are in registers: the async proxy may overwrite the buffer
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bar.uempty[h]);
                }
                if (row_ok && nvalid > 0) {
                    if constexpr (!kRes) {
                        if (qrow) {  // natural units
                            const float back = sampling ? kLn2F : 1.0f;
#pragma unroll
                            for (int c = 0; c < 16; c += 4)
                                if (c < nvalid)
                                    *reinterpret_cast<float4*>(qrow + v0 + c) = make_float4(
                                        sv[c] * back, sv[c + 1] * back, sv[c + 2] * back, sv[c + 3] * back);
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
                            // sampling draft in base 2: w = 2^(s2 - m2) relative to the running max
                            float cm = sv[0];
#pragma unroll
                            for (int c = 1; c < 16; ++c) cm = fmaxf(cm, sv[c]);
                            if (cm > part.m) {
                                const float sc = ex2(part.m - cm);  // 0 while the max is -inf
                                part.sum *= sc;
                                bw *= sc;
                                part.m = cm;
                            }
                            rho = race_bound(bE, bw);
                            uint4 x[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                x[q] = make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)pos, (uint32_t)rr, w3);
                            philox4x32_10_x4(x, key0, key1);
                            // every weight into the normaliser; entries that may beat the
                            // running winner marked for the exact test
                            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            uint32_t cand = 0;
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const uint32_t wd = word_of(x[c >> 2], c & 3);
                                const float w = ex2(sv[c] - part.m);
                                acc[c & 3] += w;
                                cand |= (one_plus_complement(wd) < fmaf(w, rho, 1.0f)) ? (1u << c) : 0u;
                            }
                            part.sum += (acc[0] + acc[1]) + (acc[2] + acc[3]);
                            if (cand) {
#pragma unroll
                                for (int c = 0; c < 16; ++c) {
                                    if (cand & (1u << c)) {
                                        const float w = ex2(sv[c] - part.m);
                                        const float E = neg_log_uniform(word_of(x[c >> 2], c & 3));
                                        if (w * bE > bw * E) {
                                            bw = w; bE = E; part.idx = v0 + c; part.s_at = sv[c];
                                            rho = race_bound(bE, bw);
                                        }
                                    }
                                }
                            }
                        }
                    } else {
                        // one race per request: over max(0, p - q) for a rejected row,
                        // over p for a bonus draw (q = 0 there)
                        if (with_u) {
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const uint32_t word = uw[c >> 1];
                                const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                                sv[c] = (u + sv[c]) * c2;
                            }
                        }
                        uint4 x[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            x[q] = make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)pos, (uint32_t)rr, w3);
                        philox4x32_10_x4(x, key0, key1);
                        {
                            const float g = fmaxf(fmaxf(g_own, g_glob),
                                                  fmaxf(fmaxf(gsh[0], gsh[kM]), fmaxf(gsh[2 * kM], gsh[3 * kM])));
                            rho = fminf(race_bound(bE, bw), ex2(-g) * kRaceSlack);
                        }
                        uint32_t cand = 0;
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float pv = ex2(fmaf(tv[c], c2, -rinfo.lse2_p));
                            const float wgt = with_u ? pv - ex2(sv[c] - rinfo.q_lse2) : pv;
                            tv[c] = wgt;
                            cand |= (wgt > 0.0f && one_plus_complement(word_of(x[c >> 2], c & 3)) <
                                                       fmaf(wgt, rho, 1.0f))
                                        ? (1u << c)
                                        : 0u;
                        }
                        if (cand) {
                            bool rec = false;
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                if (cand & (1u << c)) {
                                    const float E = neg_log_uniform(word_of(x[c >> 2], c & 3));
                                    if (tv[c] * bE > bw * E) {
                                        bw = tv[c]; bE = E; part.idx = v0 + c;
                                        rho = fminf(rho, race_bound(bE, bw));
                                        rec = true;
                                    }
                                }
                            }
                            if (rec) {
                                g_own = lg2(bw) - lg2(bE);
                                gsh[quarter * kM] = g_own;
                            }
                        }
                    }
                }
            }
            // this thread's record, if it beats the request's best seen so far, for the
            // other CTAs racing over it (few threads qualify after the first tiles:
            // same-address atomics serialise)
            if (share && g_own > fmaxf(g_pub, g_glob)) {
                const float sc = kRes ? logf(bw) - logf(bE) : part.s_at * kLn2F - logf(bE);
                atomicMax(my_key, winner_key(sc, part.idx));
                g_pub = g_own;
            }
        }
        // scores of the winners in log form, for merging across threads and CTAs
        if (kRes) {
            part.score = part.idx != INT_MAX ? logf(bw) - logf(bE) : -INFINITY;
        } else if (!p.greedy) {
            // back to natural units: the max and the winner's logit
            part.m *= kLn2F;
            part.s_at *= kLn2F;
            if (part.idx != INT_MAX) part.score = part.s_at - logf(bE);
        }
    }

    // ---------------------------------------------------------------- per-CTA result
    __syncthreads();
    TcPartial* scratch = reinterpret_cast<TcPartial*>(sB);  // W2 stages are drained
    if (warp >= kCtlWarps + 4) {
        const int m = (warp & 3) * 32 + lane;
        const int qtr = (warp - kCtlWarps) >> 2;  // 1..3
        scratch[(qtr - 1) * kM + m] = part;
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (*abort_flag) {
        if (threadIdx.x == 0) report(p.dev_status, DSPARK_ERR_TIMEOUT);
        return;
    }
    if (warp >= kCtlWarps && warp < kCtlWarps + 4 && row_ok) {
        const int m = (warp & 3) * 32 + lane;
        const int rr = row0 + m;
#pragma unroll
        for (int q = 0; q < 3; ++q) merge_any<kRes>(part, scratch[q * kM + m]);
        if (kRes) {
            if (part.idx != INT_MAX) atomicMax(p.keys + rr, winner_key(part.score, part.idx));
        } else {
            const size_t slot = (size_t)p.k * p.R + rr;
            if (!p.greedy)
                p.parts[slot * p.P + cidx] = make_float4(part.m, part.sum, part.s_at, __int_as_float(part.idx));
            if (part.idx != INT_MAX) atomicMax(p.keys + slot, winner_key(part.score, part.idx));
        }
    }
}

struct DraftFinalize {
    const unsigned long long* keys;
    const float4* parts;
    int R, gamma, P, greedy;
    int32_t* y;
    float* q_lse;
    float* q_tok;
    int32_t* dev_status;
};

// One warp per (position, request): the token from the step's winner key, the
// log-normaliser from the CTAs' (max, sum) pieces, q(y) from the piece of the
// CTA that held the winner.  A request without a key had an unusable anchor or
// predecessor (or no finite logit): its token is -1 and its q values NaN.
__global__ void __launch_bounds__(256) draft_finalize_kernel(DraftFinalize f) {
    griddep_wait();
    const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= f.R * f.gamma) return;
    const int k = gw / f.R, r = gw - k * f.R;
    const size_t slot = (size_t)k * f.R + r;
    const size_t rk = (size_t)r * f.gamma + k;
    const unsigned long long key = f.keys[slot];
    if (key == 0) {
        if (lane == 0) {
            f.y[rk] = -1;
            if (!f.greedy) {
                if (f.q_lse) f.q_lse[rk] = NAN;
                if (f.q_tok) f.q_tok[rk] = NAN;
            }
            report(f.dev_status, DSPARK_ERR_DEVICE_INPUT);
        }
        return;
    }
    const int idx = key_index(key);
    if (f.greedy) {
        if (lane == 0) f.y[rk] = idx;
        return;
    }
    float m = -INFINITY, s = 0.0f, sat = -INFINITY;
    for (int j = lane; j < f.P; j += 32) {
        const float4 q = f.parts[slot * f.P + j];
        lse_merge(m, s, q.x, q.y);
        if (__float_as_int(q.w) == idx) sat = q.z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = shfl_xor(m, o), s2 = shfl_xor(s, o);
        lse_merge(m, s, m2, s2);
        sat = fmaxf(sat, shfl_xor(sat, o));
    }
    if (lane == 0) {
        const float lse = m + logf(s);
        f.y[rk] = idx;
        if (f.q_lse) f.q_lse[rk] = lse;
        if (f.q_tok) f.q_tok[rk] = expf(sat - lse);
    }
}

// The extra token of every request, one CTA each: the race's winner (over
// max(0, p - q) for a rejected row, over p for a bonus draw).  When a rejected
// row's residual has no positive mass (p <= q everywhere), the CTA draws from
// p of the row with the same noise.
__global__ void __launch_bounds__(256) residual_finalize_kernel(const ResRow* rows, const unsigned long long* keys,
                                                                const float* target, const uint64_t* seeds,
                                                                float invT, int gamma, int V, int32_t* out_tokens,
                                                                int32_t* dev_status) {
    __shared__ unsigned long long s_key;
    const int r = blockIdx.x;
    const ResRow ri = rows[r];
    if (ri.mode == 0) return;
    unsigned long long key = keys[r];
    if (key == 0 && ri.mode == 1) {
        if (threadIdx.x == 0) s_key = 0;
        __syncthreads();
        const float c2 = invT * kLog2eF;
        const float* trow = target + (size_t)ri.trow * V;
        const uint64_t seed = seeds[r];
        float bw = 0.0f, bE = 1.0f;
        int bi = INT_MAX;
        for (int v4 = threadIdx.x; 4 * v4 < V; v4 += blockDim.x) {
            const uint4 x = philox4x32_10(make_uint4((uint32_t)v4, (uint32_t)ri.pos, (uint32_t)r, ri.w3),
                                          (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 4 * v4 + e;
                if (v >= V) break;
                const float pv = ex2(fmaf(__ldg(trow + v), c2, -ri.lse2_p));
                const float E = neg_log_uniform(word_of(x, e));
                if (pv * bE > bw * E) { bw = pv; bE = E; bi = v; }
            }
        }
        if (bi != INT_MAX) atomicMax(&s_key, winner_key(logf(bw) - logf(bE), bi));
        __syncthreads();
        key = s_key;
    }
    if (threadIdx.x == 0) {
        const int tok = key ? key_index(key) : -1;
        if (tok < 0) report(dev_status, DSPARK_ERR_DEVICE_INPUT);  // no finite score (NaN logits)
        out_tokens[(size_t)r * (gamma + 1) + ri.pos] = tok;
    }
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

// Workspace: winner keys, the A matrix H, then (draft) the A rows' tokens and
// the per-CTA normaliser pieces or (residual) the per-request rows.
struct TcLayout {
    size_t keys, n_keys, h, toks, parts, rows, total;
};
TcLayout tc_layout(int R, int gamma, int rank, bool residual) {
    TcLayout L;
    size_t off = 0;
    L.n_keys = residual ? (size_t)R : (size_t)gamma * R;
    L.keys = off; off += up256(sizeof(unsigned long long) * L.n_keys);
    L.h = off; off += up256((size_t)R * rank * 2);
    L.toks = off; off += residual ? 0 : up256(sizeof(int32_t) * (size_t)R);
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
int prepare(EncodeTiled enc, const void* U, const void* W1, const void* W2, const void* H, int R, int gamma, int V,
            int rank, bool residual, TcParams& p, CUtensorMap& tm_w2, CUtensorMap& tm_u, CUtensorMap& tm_h,
            int& grid, size_t& smem, int& n_sm) {
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int nkb = rank / kKB;
    const size_t fixed = 1024 + (size_t)nkb * kTileBytes + (residual ? 0 : 2 * (size_t)kUBufBytes) + sizeof(Bars);
    if ((size_t)max_smem < fixed + 2 * kTileBytes) return DSPARK_ERR_UNSUPPORTED;
    const int n_stages = (int)std::min<size_t>(kMaxStages, ((size_t)max_smem - fixed) / kTileBytes);
    smem = fixed + (size_t)n_stages * kTileBytes;
    // the end-of-launch exchange of the epilogue quarters reuses the drained stages
    if ((size_t)n_stages * kTileBytes < (size_t)3 * kM * sizeof(TcPartial)) return DSPARK_ERR_UNSUPPORTED;

    if (!encode_2d_bf16(enc, &tm_w2, W2, rank, V, kNV)) return DSPARK_ERR_CUDA;
    if (!encode_2d_bf16(enc, &tm_h, H, rank, R, kM)) return DSPARK_ERR_CUDA;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)R};
        const cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)gamma * V * 2};
        const cuuint32_t box[3] = {kKB, 1, kM};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tm_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_CUDA;
    }
    p = TcParams();
    p.U = static_cast<const uint16_t*>(U);
    p.W1 = static_cast<const uint16_t*>(W1);
    p.R = R;
    p.gamma = gamma;
    p.V = V;
    p.rank = rank;
    p.nb = (R + kM - 1) / kM;
    p.n_tiles = (V + kNV - 1) / kNV;
    p.P = std::max(1, std::min(std::min(n_sm / p.nb, p.n_tiles), kMaxP));
    p.n_stages = n_stages;
    p.nkb = nkb;
    grid = p.P * p.nb;
    return DSPARK_OK;
}

}  // namespace

bool draft_tc_supported(int u_dtype, int w_dtype, int R, int V, int rank) {
    return u_dtype == DSPARK_BF16 && w_dtype == DSPARK_BF16 && R >= 1 && rank % kKB == 0 && rank >= kKB &&
           rank <= 512 && V % 8 == 0 && V >= 8;
}

size_t draft_tc_workspace(int R, int gamma, int rank) { return tc_layout(R, gamma, rank, false).total; }

size_t residual_tc_workspace(int R, int rank) { return tc_layout(R, 0, rank, true).total; }

int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    if (a.q_logits && (reinterpret_cast<uintptr_t>(a.q_logits) & 15)) return DSPARK_ERR_UNSUPPORTED;
    const TcLayout L = tc_layout(a.R, a.gamma, a.rank, false);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
    uint16_t* H = reinterpret_cast<uint16_t*>(w + L.h);
    int32_t* toks = reinterpret_cast<int32_t*>(w + L.toks);
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_h;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st =
        prepare(enc, a.U, a.W1, a.W2, H, a.R, a.gamma, a.V, a.rank, false, p, tm_w2, tm_u, tm_h, grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    p.keys = reinterpret_cast<unsigned long long*>(w + L.keys);
    p.toks = toks;
    p.parts = reinterpret_cast<float4*>(w + L.parts);
    p.anchor = a.anchor;
    p.seeds = a.seeds;
    p.q_logits = a.q_logits;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = a.greedy;
    if (cudaFuncSetAttribute(markov_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(p.keys, 0, sizeof(unsigned long long) * L.n_keys, stream) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    // gather 0 waits for everything before it on the stream.  Every later launch
    // is a programmatic dependent of the one before: it may start as that one
    // retires and waits (griddepcontrol) before reading its results; the only
    // data read earlier are W2 and U.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchConfig_t gcfg = {};
    gcfg.gridDim = dim3((unsigned)a.R);
    gcfg.blockDim = dim3(kGatherThreads);
    gcfg.stream = stream;
    gcfg.attrs = attr;
    for (int k = 0; k < a.gamma; ++k) {
        gcfg.numAttrs = k == 0 ? 0 : 1;
        const unsigned long long* prev_keys = k == 0 ? nullptr : p.keys + (size_t)(k - 1) * a.R;
        if (cudaLaunchKernelEx(&gcfg, gather_a_rows_kernel, p.W1, a.anchor, prev_keys, k, a.R, a.V, a.rank, H,
                               toks) != cudaSuccess)
            return DSPARK_ERR_CUDA;
        p.k = k;
        if (cudaLaunchKernelEx(&cfg, markov_tc_kernel<false>, tm_w2, tm_u, tm_h, p) != cudaSuccess)
            return DSPARK_ERR_CUDA;
    }
    DraftFinalize f;
    f.keys = p.keys;
    f.parts = p.parts;
    f.R = a.R;
    f.gamma = a.gamma;
    f.P = p.P;
    f.greedy = a.greedy;
    f.y = a.y;
    f.q_lse = a.q_lse;
    f.q_tok = a.q_tok;
    f.dev_status = a.dev_status;
    cudaLaunchConfig_t fcfg = {};
    const long long warps = (long long)a.R * a.gamma;
    fcfg.gridDim = dim3((unsigned)((warps * 32 + 255) / 256));
    fcfg.blockDim = dim3(256);
    fcfg.stream = stream;
    fcfg.attrs = attr;
    fcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&fcfg, draft_finalize_kernel, f) != cudaSuccess) return DSPARK_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int launch_residual_tc(const ResidualTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    const TcLayout L = tc_layout(a.R, a.gamma, a.rank, true);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
    uint16_t* H = reinterpret_cast<uint16_t*>(w + L.h);
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_h;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st =
        prepare(enc, a.U, a.W1, a.W2, H, a.R, a.gamma, a.V, a.rank, true, p, tm_w2, tm_u, tm_h, grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    ResRow* rows = reinterpret_cast<ResRow*>(w + L.rows);
    p.keys = reinterpret_cast<unsigned long long*>(w + L.keys);
    p.anchor = a.anchor;
    p.seeds = a.seeds;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = 0;
    p.target = a.target;
    p.rows = rows;
    p.k = 0;
    if (cudaFuncSetAttribute(markov_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(p.keys, 0, sizeof(unsigned long long) * L.n_keys, stream) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    residual_prep_kernel<<<(unsigned)((a.R * 32LL + 255) / 256), 256, 0, stream>>>(a, rows, H);
    markov_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tm_w2, tm_u, tm_h, p);
    residual_finalize_kernel<<<a.R, 256, 0, stream>>>(rows, p.keys, a.target, a.seeds, a.invT, a.gamma, a.V,
                                                      a.out_tokens, a.dev_status);
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark

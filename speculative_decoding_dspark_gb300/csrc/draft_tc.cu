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
// Persistent, one CTA per SM, 18 warps:
//   A (M = 128 requests x K = rank) = rows W1[prev], gathered by the epilogue
//     warps straight into 128-byte-swizzled shared memory at the start of the
//     launch and resident for it;
//   B (N = 128 vocabulary rows x K = rank) = W2 tiles streamed by TMA through a
//     ring of 16 KB stages; the next tile's boxes are prefetched into L2 one
//     tile ahead so the ring only has to cover L2 latency;
//   D = A . B^T in fp32 tensor memory, two 128-column buffers so the epilogue
//     of one vocabulary tile overlaps the MMAs of the next;
//   epilogue (16 warps; thread = one request x 32 vocabulary columns, in two
//     16-column passes): Gumbel-max draws use the exponential-race form: with
//     weight w > 0 and E = -log(u), the largest log(w) + Gumbel(u) is the
//     largest w / E, so a candidate replaces the best when
//     w * E_best > w_best * E.  Since E >= 1 - u, an entry with
//     1 - u >= w * E_best / w_best cannot win; that test needs no logarithm
//     (1 - u comes exactly from the random bits), and only the entries that
//     pass it take the accurate log and the exact comparison.
//
// Cross-CTA results need no merging pass: every CTA folds its winner into one
// 64-bit key per request and step with atomicMax (order-preserving bits of
// the score above the inverted index, so ties go to the lower index), and
// stores its (max, sum of exp, winner logit) piece of the normaliser.  The
// next draft step decodes its A rows' tokens from the keys (it is launched
// as a programmatic dependent and waits for the previous step before reading
// them, while its producer already streams W2), and one finalize kernel after
// the last step turns keys and pieces into tokens, q_lse and q(y).
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2-17 = A gather, then epilogue.  Every mbarrier wait is bounded (2 s);
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
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kCols = 32;                     // vocabulary columns per epilogue thread
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
// (score, idx) over the residual, (s_at, m-as-index) the draw over p.
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
    unsigned long long* keys;  // draft [gamma][R]; residual [2][R] (residual race, p race)
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
    uint64_t afull, mma_done;
    uint32_t tmem_slot;
    int abort_flag;
    int tok[kM];  // token of each A row: >= 0 a W1 row, -1 zero row, -2 zero row and no result
};

__device__ __forceinline__ void merge_draft(float& sc, int& ix, float& sa, float& m, float& su, float sc2, int ix2,
                                            float sa2, float m2, float su2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; sa = sa2; }
    lse_merge(m, su, m2, su2);
}

__device__ __forceinline__ void merge_residual(float& sc, int& ix, float& sa, int& ia, float sc2, int ix2, float sa2,
                                               int ia2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; }
    if (better(sa2, ia2, sa, ia)) { sa = sa2; ia = ia2; }
}

template <bool kRes>
__device__ __forceinline__ void merge_any(TcPartial& a, const TcPartial& b) {
    if (kRes) {
        int ia = __float_as_int(a.m);
        merge_residual(a.score, a.idx, a.s_at, ia, b.score, b.idx, b.s_at, __float_as_int(b.m));
        a.m = __int_as_float(ia);
    } else {
        merge_draft(a.score, a.idx, a.s_at, a.m, a.sum, b.score, b.idx, b.s_at, b.m, b.sum);
    }
}

template <bool kRes>
__device__ __forceinline__ TcPartial identity_partial() {
    TcPartial w;
    w.score = -INFINITY; w.idx = INT_MAX; w.s_at = kRes ? -INFINITY : 0.0f;
    w.m = kRes ? __int_as_float(INT_MAX) : -INFINITY; w.sum = 0.0f;
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

// 1 + (1 - u) - 2^-24 for u = uniform_from_bits(x): the 23 kept bits inverted
// under the exponent of 1.0 (exact).
__device__ __forceinline__ float one_plus_complement(uint32_t x) {
    return __uint_as_float((x >> 9) ^ 0x3FFFFFFFu);
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

__device__ __forceinline__ void epilogue_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// Per request after the verify decisions: what the residual launch draws and
// the token whose W1 row is its A row (the rejected position's predecessor).
__global__ void __launch_bounds__(256) residual_prep_kernel(ResidualTcArgs a, ResRow* rows) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
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
    rows[r] = w;
}

template <bool kRes>
__global__ void __launch_bounds__(kThreads, 1)
markov_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
                 const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + p.nkb * kTileBytes;
    Bars& bar = *reinterpret_cast<Bars*>(sB + p.n_stages * kTileBytes);
    volatile int* abort_flag = &bar.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = blockIdx.x % p.nb;
    const int cidx = blockIdx.x / p.nb;
    const int row0 = blk * kM;
    const int S = p.n_stages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { tc::mbar_init(&bar.full[s], 1); tc::mbar_init(&bar.empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar.tfull[a], 1); tc::mbar_init(&bar.tempty[a], kEpiWarps); }
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
        // W2 and U are inputs no launch of this library writes, so streaming
        // them may start before the previous draft step has finished.
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int last_phase[kMaxStages];
            for (int i = 0; i < kMaxStages; ++i) last_phase[i] = -1;
            bool ok = true;
            for (int i = 0; i < 2 && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                for (int q = 0; q < p.nkb; ++q) tma_prefetch_l2_2d(&tm_w2, q * kKB, t * kNV);
                if (!kRes) {
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV, p.k, row0);
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV + kKB, p.k, row0);
                }
            }
            for (int i = 0; ok && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(&bar.full[s], kTileBytes);
                    tc::tma_load_2d(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV);
                    last_phase[s] = (int)ph;
                    if (++s == S) { s = 0; ph ^= 1u; }
                    // once this tile's first loads are out, pull the next tile into L2
                    if (kb == min(S, p.nkb) - 1 && i + 1 < n_local) {
                        const int tn = t + p.P;
                        for (int q = 0; q < p.nkb; ++q) tma_prefetch_l2_2d(&tm_w2, q * kKB, tn * kNV);
                        if (!kRes) {
                            tc::tma_prefetch_l2_3d(&tm_u, tn * kNV, p.k, row0);
                            tc::tma_prefetch_l2_3d(&tm_u, tn * kNV + kKB, p.k, row0);
                        }
                    }
                }
            }
            // after an abort, the copies this thread issued must land before the CTA exits
            if (*abort_flag) {
                int dummy = 0;
                volatile int* no_abort = &dummy;
                for (int q = 0; q < S; ++q)
                    if (last_phase[q] >= 0) tc::mbar_wait(&bar.full[q], (uint32_t)last_phase[q], no_abort, kWaitNs);
            }
        }
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
    } else {
        // ------------------------------------------------------------ A gather
        const int et = threadIdx.x - 64;  // 0..511
        // the previous draft step's winners are read after this
        griddep_wait();
        if (et < kM) {
            const int r = row0 + et;
            int t = -1;
            if (r < p.R) {
                if (kRes) {
                    const ResRow ri = p.rows[r];
                    t = ri.mode == 0 ? -2 : ri.prev;
                } else if (p.k == 0) {
                    const int a = p.anchor[r];
                    t = a >= p.V ? -2 : (a < 0 ? -1 : a);
                } else {
                    const unsigned long long key = __ldcg(p.keys + (size_t)(p.k - 1) * p.R + r);
                    t = key ? key_index(key) : -2;
                }
            } else {
                t = -2;
            }
            bar.tok[et] = t;
        }
        epilogue_barrier();
        {
            // A row m, k-block kb, 16-byte chunk j sits at chunk j ^ (m & 7) of its
            // 128-byte row: the layout a 128-byte-swizzled TMA box would give.
            const int cpr = p.rank >> 3;
            const int total = kM * cpr;
            for (int e0 = et; e0 < total; e0 += 8 * kEpiThreads) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + u * kEpiThreads;
                    v[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (e < total) {
                        const int m = e / cpr, c = e - m * cpr;
                        const int t = bar.tok[m];
                        if (t >= 0) v[u] = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)t * p.rank) + c);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + u * kEpiThreads;
                    if (e < total) {
                        const int m = e / cpr, c = e - m * cpr;
                        const int off = (c >> 3) * kTileBytes + m * 128 + (((c & 7) ^ (m & 7)) << 4);
                        *reinterpret_cast<uint4*>(sA + off) = v[u];
                    }
                }
            }
        }
        // the tensor cores read A through the async proxy
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar.afull);

        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;           // 0..15
        const int quad = warp & 3;         // TMEM lane quadrant this warp may read
        const int quarter = ew >> 2;       // which 32 of the tile's 128 columns
        const int m = quad * 32 + lane;
        const int rr = row0 + m;
        row_ok = bar.tok[m] != -2;
        ResRow rinfo;
        rinfo.mode = 0; rinfo.pos = 0; rinfo.trow = 0; rinfo.w3 = 0; rinfo.lse2_p = 0.0f; rinfo.q_lse2 = 0.0f;
        if (kRes && row_ok) rinfo = p.rows[rr];
        const bool sampling = kRes || !p.greedy;
        PhiloxKey K;
        if (sampling) K = philox_key(row_ok ? p.seeds[rr] : 0ull);
        const uint32_t w3 = kRes ? rinfo.w3 : ctr_word3(p.cycle, kDraftGumbel);
        const int pos = kRes ? rinfo.pos : p.k;
        const bool with_u = !kRes || rinfo.mode == 1;
        const size_t rk = (size_t)rr * p.gamma + pos;
        const uint16_t* urow = p.U + rk * p.V;
        const float* trow = kRes ? p.target + (size_t)rinfo.trow * p.V : nullptr;
        float* qrow = (!kRes && p.q_logits && row_ok) ? p.q_logits + rk * p.V : nullptr;
        // logits are scaled to base 2 when sampling: s2 = s * log2(e) / T
        const float c2 = sampling ? p.invT * kLog2eF : 1.0f;
        // exponential-race state: draft / residual race (bw, bE, rho), p race (bp, bEp, rho_p);
        // rho = E_best / w_best with the slack, the bound of the no-log test
        float bw = 0.0f, bE = 1.0f, bp = 0.0f, bEp = 1.0f;
        float rho = INFINITY, rho_p = INFINITY;
        int ia = INT_MAX;
        for (int i = 0; i < n_local; ++i) {
            const int t = cidx + i * p.P;
            const int a = i & 1;
            const uint32_t use = (uint32_t)(i >> 1);
            const int vq = t * kNV + quarter * kCols;
            uint32_t uwA[8], uwB[8];
            if (!kRes) {
                // base logits of this thread's 32 columns (already in L2), two halves
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint4 qa = (row_ok && 8 * j < p.V - vq) ? __ldg(reinterpret_cast<const uint4*>(urow + vq) + j)
                                                                  : make_uint4(0u, 0u, 0u, 0u);
                    const uint4 qb = (row_ok && 16 + 8 * j < p.V - vq)
                                         ? __ldg(reinterpret_cast<const uint4*>(urow + vq) + 2 + j)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    uwA[4 * j + 0] = qa.x; uwA[4 * j + 1] = qa.y; uwA[4 * j + 2] = qa.z; uwA[4 * j + 3] = qa.w;
                    uwB[4 * j + 0] = qb.x; uwB[4 * j + 1] = qb.y; uwB[4 * j + 2] = qb.z; uwB[4 * j + 3] = qb.w;
                }
            } else if (row_ok && vq < p.V) {
                // residual rows differ per request: pull this thread's pieces into L2 now
                prefetch_l2(trow + vq);
                if (with_u) prefetch_l2(urow + vq);
            }
            // warp-uniform wait: every lane waits (acquire), all leave together
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar.tfull[a], use & 1u, abort_flag, kWaitNs))) break;
            tc::tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * kNV + quarter * kCols);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float sv[16];
                __syncwarp();  // lanes that skipped the previous pass rejoin before the aligned load
                tc::tmem_ld_32x32b_x16<0>(taddr + 16u * h, sv);
                tc::tmem_ld_wait();
                if (h == 1) {  // both halves are in registers: hand the accumulator back
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bar.tempty[a]);
                }
                if (!row_ok) continue;
                const int v0 = vq + 16 * h;
                const int nvalid = min(16, p.V - v0);
                if (kRes && with_u) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint4 q4 = 8 * j < nvalid ? __ldg(reinterpret_cast<const uint4*>(urow + v0) + j)
                                                        : make_uint4(0u, 0u, 0u, 0u);
                        uwA[4 * j + 0] = q4.x; uwA[4 * j + 1] = q4.y; uwA[4 * j + 2] = q4.z; uwA[4 * j + 3] = q4.w;
                    }
                }
                if (!kRes || with_u) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint32_t word = (kRes || h == 0) ? uwA[c >> 1] : uwB[c >> 1];
                        const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                        sv[c] = (u + sv[c]) * c2;
                    }
                }
                if (qrow) {  // natural units
                    const float back = sampling ? kLn2F : 1.0f;
#pragma unroll
                    for (int c = 0; c < 16; c += 4)
                        if (c < nvalid)
                            *reinterpret_cast<float4*>(qrow + v0 + c) =
                                make_float4(sv[c] * back, sv[c + 1] * back, sv[c + 2] * back, sv[c + 3] * back);
                }
                if (!kRes && p.greedy) {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c < nvalid && better(sv[c], v0 + c, part.score, part.idx)) {
                            part.score = sv[c]; part.idx = v0 + c; part.s_at = sv[c];
                        }
                    continue;
                }
                if constexpr (!kRes) {
                    // sampling draft in base 2: w = 2^(s2 - m2) relative to the running max
                    float cm = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c < nvalid) cm = fmaxf(cm, sv[c]);
                    if (cm > part.m) {
                        const float sc = ex2(part.m - cm);  // 0 while the max is -inf
                        part.sum *= sc;
                        bw *= sc;
                        part.m = cm;
                        rho = bE / bw * kRaceSlack;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 wd = philox4x32_10(
                            make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)pos, (uint32_t)rr, w3), K);
                        const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * q + e;
                            if (c < nvalid) {
                                const float w = ex2(sv[c] - part.m);
                                part.sum += w;
                                if (one_plus_complement(words[e]) < fmaf(w, rho, 1.0f)) {
                                    const float E = -logf(uniform_from_bits(words[e]));
                                    if (w * bE > bw * E) {
                                        bw = w; bE = E; part.idx = v0 + c; part.s_at = sv[c];
                                        rho = bE / bw * kRaceSlack;
                                    }
                                }
                            }
                        }
                    }
                } else {
                    float tv[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 f = 4 * j < nvalid ? __ldg(reinterpret_cast<const float4*>(trow + v0) + j)
                                                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        tv[4 * j + 0] = f.x; tv[4 * j + 1] = f.y; tv[4 * j + 2] = f.z; tv[4 * j + 3] = f.w;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 wd = philox4x32_10(
                            make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)pos, (uint32_t)rr, w3), K);
                        const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * q + e;
                            if (c < nvalid) {
                                const float pv = ex2(fmaf(tv[c], c2, -rinfo.lse2_p));
                                const float res = with_u ? pv - ex2(sv[c] - rinfo.q_lse2) : 0.0f;
                                const float f = one_plus_complement(words[e]);
                                const bool try_p = f < fmaf(pv, rho_p, 1.0f);
                                const bool try_r = res > 0.0f && f < fmaf(res, rho, 1.0f);
                                if (try_p || try_r) {
                                    const float E = -logf(uniform_from_bits(words[e]));
                                    if (try_p && pv * bEp > bp * E) {
                                        bp = pv; bEp = E; ia = v0 + c;
                                        rho_p = bEp / bp * kRaceSlack;
                                    }
                                    if (try_r && res * bE > bw * E) {
                                        bw = res; bE = E; part.idx = v0 + c;
                                        rho = bE / bw * kRaceSlack;
                                    }
                                }
                            }
                        }
                    }
                }
            }
        }
        // scores of the winners in log form, for merging across threads and CTAs
        if (kRes) {
            part.score = part.idx != INT_MAX ? logf(bw) - logf(bE) : -INFINITY;
            part.s_at = ia != INT_MAX ? logf(bp) - logf(bEp) : -INFINITY;
            part.m = __int_as_float(ia);
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
    if (warp >= 6) {
        const int m = (warp & 3) * 32 + lane;
        const int qtr = (warp - 2) >> 2;  // 1..3
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
    if (warp >= 2 && warp < 6 && row_ok) {
        const int m = (warp & 3) * 32 + lane;
        const int rr = row0 + m;
#pragma unroll
        for (int q = 0; q < 3; ++q) merge_any<kRes>(part, scratch[q * kM + m]);
        if (kRes) {
            if (part.idx != INT_MAX) atomicMax(p.keys + rr, winner_key(part.score, part.idx));
            const int ia = __float_as_int(part.m);
            if (ia != INT_MAX) atomicMax(p.keys + p.R + rr, winner_key(part.s_at, ia));
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

// The extra token of every request: the residual winner when the residual has
// mass (mode 1), else the winner over p.
__global__ void __launch_bounds__(256) residual_finalize_kernel(const ResRow* rows, const unsigned long long* keys,
                                                                int R, int gamma, int32_t* out_tokens,
                                                                int32_t* dev_status) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const ResRow ri = rows[r];
    if (ri.mode == 0) return;
    const unsigned long long kr = keys[r], kp = keys[R + r];
    int tok = -1;
    if (ri.mode == 1 && kr) tok = key_index(kr);
    else if (kp) tok = key_index(kp);
    if (tok < 0) report(dev_status, DSPARK_ERR_DEVICE_INPUT);  // no finite score (NaN logits)
    out_tokens[(size_t)r * (gamma + 1) + ri.pos] = tok;
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

// Workspace: winner keys, then (draft) the per-CTA normaliser pieces or
// (residual) the per-request rows.
struct TcLayout {
    size_t keys, n_keys, parts, rows, total;
};
TcLayout tc_layout(int R, int gamma, bool residual) {
    TcLayout L;
    size_t off = 0;
    L.n_keys = residual ? 2 * (size_t)R : (size_t)gamma * R;
    L.keys = off; off += up256(sizeof(unsigned long long) * L.n_keys);
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
int prepare(EncodeTiled enc, const void* U, const void* W1, const void* W2, int R, int gamma, int V, int rank,
            TcParams& p, CUtensorMap& tm_w2, CUtensorMap& tm_u, int& grid, size_t& smem, int& n_sm) {
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int nkb = rank / kKB;
    const size_t fixed = 1024 + (size_t)nkb * kTileBytes + sizeof(Bars);
    if ((size_t)max_smem < fixed + 2 * kTileBytes) return DSPARK_ERR_UNSUPPORTED;
    const int n_stages = (int)std::min<size_t>(kMaxStages, ((size_t)max_smem - fixed) / kTileBytes);
    smem = fixed + (size_t)n_stages * kTileBytes;
    // the end-of-launch exchange of the epilogue quarters reuses the drained stages
    if ((size_t)n_stages * kTileBytes < (size_t)3 * kM * sizeof(TcPartial)) return DSPARK_ERR_UNSUPPORTED;

    if (!encode_2d_bf16(enc, &tm_w2, W2, rank, V, kNV)) return DSPARK_ERR_CUDA;
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

size_t draft_tc_workspace(int R, int gamma, int) { return tc_layout(R, gamma, false).total; }

size_t residual_tc_workspace(int R, int) { return tc_layout(R, 0, true).total; }

int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    if (a.q_logits && (reinterpret_cast<uintptr_t>(a.q_logits) & 15)) return DSPARK_ERR_UNSUPPORTED;
    TcParams p;
    CUtensorMap tm_w2, tm_u;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st = prepare(enc, a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, p, tm_w2, tm_u, grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    const TcLayout L = tc_layout(a.R, a.gamma, false);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
    p.keys = reinterpret_cast<unsigned long long*>(w + L.keys);
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
    // Step 0 waits for everything before it on the stream.  Steps 1.. and the
    // finalize are programmatic dependents of the launch before them: they may
    // start as its CTAs retire and wait (griddepcontrol) before reading its
    // results; the only data they touch earlier are W2 and U.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    for (int k = 0; k < a.gamma; ++k) {
        p.k = k;
        cfg.numAttrs = k == 0 ? 0 : 1;
        if (cudaLaunchKernelEx(&cfg, markov_tc_kernel<false>, tm_w2, tm_u, p) != cudaSuccess) return DSPARK_ERR_CUDA;
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
    TcParams p;
    CUtensorMap tm_w2, tm_u;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st = prepare(enc, a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, p, tm_w2, tm_u, grid, smem, n_sm);
    if (st != DSPARK_OK) return st;
    const TcLayout L = tc_layout(a.R, a.gamma, true);
    unsigned char* w = static_cast<unsigned char*>(a.ws);
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
    const int blocks = (a.R + 255) / 256;
    residual_prep_kernel<<<blocks, 256, 0, stream>>>(a, rows);
    markov_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tm_w2, tm_u, p);
    residual_finalize_kernel<<<blocks, 256, 0, stream>>>(rows, p.keys, a.R, a.gamma, a.out_tokens, a.dev_status);
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark

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
//             sample, log-normaliser and q(y);
//   residual  one launch per verify: for every request the drafter's logits of
//             its rejected row are recomputed here (the residual needs q on the
//             whole vocabulary, and recomputing one row per request costs one
//             pass over W2 instead of keeping every drafted row in memory),
//             then the extra token is drawn from max(0, p - q), or from p after
//             full acceptance.
//
// Persistent, one CTA per SM, 18 warps:
//   A (M = 128 requests x K = rank) = rows W1[prev] gathered into a workspace
//     matrix H (a small kernel for the anchors or the residual rows, the
//     reducer of draft step k for step k + 1), loaded by TMA into
//     128-byte-swizzled shared memory and resident for the launch;
//   B (N = 128 vocabulary rows x K = rank) = W2 tiles streamed by TMA through a
//     ring of 16 KB stages; the next tile's boxes are prefetched into L2 one
//     tile ahead so the ring only has to cover L2 latency;
//   D = A . B^T in fp32 tensor memory, two 128-column buffers so the epilogue
//     of one vocabulary tile overlaps the MMAs of the next;
//   epilogue (16 warps; thread = one request x 32 vocabulary columns, in two
//     16-column passes): Gumbel-max draws use the exponential-race form: with
//     weight w > 0 and E = -log(u), the largest log(w) + Gumbel(u) is the
//     largest w / E, so a candidate replaces the best when
//     w * E_best > w_best * E (one log per entry, no log of the weight).
// Each CTA leaves one partial per request; reduction is two-level and never
// spins: the last CTA of each group of kGroup CTAs (atomic counter) merges its
// group, the last group of a request block merges the groups.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2-17 = epilogue.  Every mbarrier wait is bounded (2 s); a timeout
// aborts the CTA cleanly and reports DSPARK_ERR_TIMEOUT.
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
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kCols = 32;                     // vocabulary columns per epilogue thread
constexpr int kMaxStages = 8;
constexpr int kMaxP = 256;                    // partials per request (>= CTAs per block)
constexpr int kGroup = 16;                    // CTAs per first-level reduction group
constexpr int kMaxGroups = kMaxP / kGroup;
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

// Per-request partial.  Draft: (score, idx) of the Gumbel-max draw, s at it,
// (max, sum of exp) of the logits.  Residual: (score, idx) over the residual,
// (s_at, m-as-index) the draw over p, sum = residual mass seen.
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
    float lse_p;   // target log-normaliser of the row (scaled logits)
    float q_lse;   // drafter log-normaliser at pos (mode 1)
    float pad[2];
};

struct TcParams {
    const uint16_t* U;
    const uint16_t* W1;
    uint16_t* H;           // [R, rank] the A rows
    int* gcount;           // [nb * kMaxGroups] first-level counters
    int* tcount;           // [nb] second-level counters
    TcPartial* parts;      // [R * kMaxP]
    TcPartial* gparts;     // [R * kMaxGroups]
    const uint64_t* seeds;
    int32_t* dev_status;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank, k;
    int nb, P, n_groups, n_tiles, n_stages, nkb;
    // draft
    const int32_t* anchor;
    int32_t* y;
    float* q_lse;
    float* q_tok;
    float* q_logits;
    // residual
    const float* target;
    const ResRow* rows;
    int32_t* out_tokens;
};

struct Bars {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t tfull[2], tempty[2];
    uint64_t afull, mma_done;
    uint32_t tmem_slot;
    int abort_flag;
    int last;
    int top;
};

__device__ __forceinline__ void merge_draft(float& sc, int& ix, float& sa, float& m, float& su, float sc2, int ix2,
                                            float sa2, float m2, float su2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; sa = sa2; }
    lse_merge(m, su, m2, su2);
}

__device__ __forceinline__ void merge_residual(float& sc, int& ix, float& sa, int& ia, float& su, float sc2, int ix2,
                                               float sa2, int ia2, float su2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; }
    if (better(sa2, ia2, sa, ia)) { sa = sa2; ia = ia2; }
    su += su2;
}

template <bool kRes>
__device__ __forceinline__ void merge_any(TcPartial& a, const TcPartial& b) {
    if (kRes) {
        int ia = __float_as_int(a.m);
        merge_residual(a.score, a.idx, a.s_at, ia, a.sum, b.score, b.idx, b.s_at, __float_as_int(b.m), b.sum);
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

__device__ __forceinline__ int prev_of(const TcParams& p, int r) {  // -1 none, -2 bad
    if (p.k == 0) {
        const int a = p.anchor[r];
        return a >= p.V ? -2 : (a < 0 ? -1 : a);
    }
    const int t = p.y[(size_t)r * p.gamma + p.k - 1];
    return (t < 0 || t >= p.V) ? -2 : t;
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on to
// complete (and their writes to be visible); allow dependents to start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Copies rows x n partials (row stride `stride`, first column `first`) into
// shared memory with every load issued before any is used: one L2 round trip.
__device__ __forceinline__ void stage_partials(TcPartial* dst, const TcPartial* src, size_t stride, int first,
                                               int n, int rows) {
    const int total = rows * n;
    for (int e0 = threadIdx.x; e0 < total; e0 += 4 * kThreads) {
        float4 lo[4], hi[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) {
                const int r = e / n, j = e - r * n;
                const float4* q = reinterpret_cast<const float4*>(src + (size_t)r * stride + first + j);
                lo[u] = __ldcg(q);
                hi[u] = __ldcg(q + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) {
                reinterpret_cast<float4*>(dst + e)[0] = lo[u];
                reinterpret_cast<float4*>(dst + e)[1] = hi[u];
            }
        }
    }
}

// H[r] = W1[anchor[r]] (zeros when there is no usable anchor): the A rows of draft step 0.
__global__ void __launch_bounds__(256) gather_anchor_rows_kernel(const uint16_t* W1, const int32_t* anchor,
                                                                 int R, int V, int rank, uint16_t* H) {
    const int cpr = rank >> 3;  // 16-byte chunks per row
    const long long total = (long long)R * cpr;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(e / cpr), c = (int)(e - (long long)r * cpr);
        const int a = anchor[r];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (a >= 0 && a < V) v = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)a * rank) + c);
        reinterpret_cast<uint4*>(H + (size_t)r * rank)[c] = v;
    }
}

// Per request after the verify decisions: what the residual launch draws, and
// its A row W1[prev] of the rejected position (zeros for a bonus draw).
__global__ void __launch_bounds__(256) residual_prep_kernel(ResidualTcArgs a, ResRow* rows, uint16_t* H) {
    const int cpr = a.rank >> 3;
    const long long total = (long long)a.R * cpr;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(e / cpr), c = (int)(e - (long long)r * cpr);
        const VerifyJob job = a.jobs[r];
        const int mode = a.valid[r] ? job.mode : 0;
        int prev = -1;
        if (mode == 1) {
            prev = job.pos == 0 ? a.anchor[r] : a.y[(size_t)r * a.gamma + job.pos - 1];
            if (prev >= a.V) prev = -1;
        }
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (prev >= 0) v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.W1) + (size_t)prev * a.rank) + c);
        reinterpret_cast<uint4*>(H + (size_t)r * a.rank)[c] = v;
        if (c == 0) {
            ResRow w;
            w.mode = mode;
            w.pos = job.pos;
            w.trow = job.row;
            w.w3 = ctr_word3(a.cycle, mode == 1 ? kResidualGumbel : kBonusGumbel);
            w.lse_p = job.lse;
            w.q_lse = mode == 1 ? a.q_lse[(size_t)r * a.gamma + job.pos] : 0.0f;
            w.pad[0] = w.pad[1] = 0.0f;
            rows[r] = w;
        }
    }
}

template <bool kRes>
__global__ void __launch_bounds__(kThreads, 1)
markov_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
                 const __grid_constant__ CUtensorMap tm_h, const TcParams p) {
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
        tc::mbar_init(&bar.afull, 1);
        tc::mbar_init(&bar.mma_done, 1);
        bar.abort_flag = 0;
        bar.last = 0;
        bar.top = 0;
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
    const uint32_t tmem_base = bar.tmem_slot;
    const int n_local = cidx < p.n_tiles ? (p.n_tiles - 1 - cidx) / p.P + 1 : 0;

    // this thread's running partial (epilogue threads)
    TcPartial part = identity_partial<kRes>();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int last_phase[kMaxStages];
            for (int i = 0; i < kMaxStages; ++i) last_phase[i] = -1;
            bool ok = true;
            // The first tiles do not depend on the previous launch: pull them into
            // L2 while that launch may still be finishing (programmatic launch).
            for (int i = 0; i < 2 && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                for (int q = 0; q < p.nkb; ++q) tma_prefetch_l2_2d(&tm_w2, q * kKB, t * kNV);
                if (!kRes) {
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV, p.k, row0);
                    tc::tma_prefetch_l2_3d(&tm_u, t * kNV + kKB, p.k, row0);
                }
            }
            // H (and everything else the previous launch wrote) is ready after this
            griddep_wait();
            // A: the block's H rows, resident for the launch
            tc::mbar_arrive_expect_tx(&bar.afull, (uint32_t)(p.nkb * kTileBytes));
            for (int kb = 0; kb < p.nkb; ++kb) tc::tma_load_2d(sA + kb * kTileBytes, &tm_h, &bar.afull, kb * kKB, row0);
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
            // the copies this thread issued must land before the CTA exits
            int dummy = 0;
            volatile int* no_abort = &dummy;
            tc::mbar_wait(&bar.afull, 0, no_abort, kWaitNs);
            if (*abort_flag) {
                for (int q = 0; q < S; ++q)
                    if (last_phase[q] >= 0) tc::mbar_wait(&bar.full[q], (uint32_t)last_phase[q], no_abort, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kM, kNV);
            bool ok = tc::mbar_wait(&bar.afull, 0, abort_flag, kWaitNs);
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
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;           // 0..15
        const int quad = warp & 3;         // TMEM lane quadrant this warp may read
        const int quarter = ew >> 2;       // which 32 of the tile's 128 columns
        const int m = quad * 32 + lane;
        const int rr = row0 + m;
        bool row_ok = rr < p.R;
        // per-row constants of the two modes
        ResRow rinfo;
        rinfo.mode = 0; rinfo.pos = 0; rinfo.trow = 0; rinfo.w3 = 0; rinfo.lse_p = 0.0f; rinfo.q_lse = 0.0f;
        if (kRes && row_ok) {
            rinfo = p.rows[rr];
            row_ok = rinfo.mode != 0;
        }
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
        // exponential-race state: draft (bw, bE); residual (br, bEr) and (bp, bEp)
        float bw = 0.0f, bE = 1.0f, bp = 0.0f, bEp = 1.0f;
        float rho2 = INFINITY;  // draft: E_best * log2(e) / w_best
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
                        const float sb = u + sv[c];
                        sv[c] = (!kRes && p.greedy) ? sb : sb * p.invT;
                    }
                }
                if (qrow) {
#pragma unroll
                    for (int c = 0; c < 16; c += 4)
                        if (c < nvalid)
                            *reinterpret_cast<float4*>(qrow + v0 + c) = make_float4(sv[c], sv[c + 1], sv[c + 2], sv[c + 3]);
                }
                if (!kRes && p.greedy) {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c < nvalid && better(sv[c], v0 + c, part.score, part.idx)) {
                            part.score = sv[c]; part.idx = v0 + c; part.s_at = sv[c];
                        }
                    continue;
                }
                if (!kRes) {
                    // Sampling draft, base-2 units: s2 = s * log2(e), w = 2^(s2 - m2).
                    // An entry can only replace the best when w * E_best > w_best * E,
                    // i.e. u > exp(-w * E_best / w_best); that bound is tested first
                    // (with a 2^-14 relative margin against the rounding of its
                    // approximations) and the accurate log and exact comparison run
                    // only for entries that pass it.
                    float cm = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        sv[c] *= kLog2eF;
                        if (c < nvalid) cm = fmaxf(cm, sv[c]);
                    }
                    if (cm > part.m) {
                        const float sc = exp2f(part.m - cm);  // 0 while the max is -inf
                        part.sum *= sc;
                        bw *= sc;
                        part.m = cm;
                        rho2 = bE * kLog2eF / bw;
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
                                const float w = exp2f(sv[c] - part.m);
                                part.sum += w;
                                const float u = uniform_from_bits(words[e]);
                                if (u > exp2f(-w * rho2) * (1.0f - 0x1p-14f)) {
                                    const float E = -logf(u);
                                    if (w * bE > bw * E) {
                                        bw = w; bE = E; part.idx = v0 + c; part.s_at = sv[c];
                                        rho2 = bE * kLog2eF / bw;
                                    }
                                }
                            }
                        }
                    }
                    continue;
                }
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
                            const float E = -logf(uniform_from_bits(words[e]));
                            const float pv = expf(tv[c] * p.invT - rinfo.lse_p);
                            if (pv * bEp > bp * E) { bp = pv; bEp = E; ia = v0 + c; }
                            if (with_u) {
                                const float res = pv - expf(sv[c] - rinfo.q_lse);
                                if (res > 0.0f) {
                                    part.sum += res;
                                    if (res * bE > bw * E) { bw = res; bE = E; part.idx = v0 + c; }
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

    // ---------------------------------------------------------------- per-CTA partials
    // The next launch may start on SMs this grid leaves; the workspace below is
    // shared with the previous launch, so wait for it to have finished.
    griddep_launch_dependents();
    griddep_wait();
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
    const bool aborted = *abort_flag != 0;
    if (warp >= 2 && warp < 6 && !aborted) {
        const int m = (warp & 3) * 32 + lane;
        const int rr = row0 + m;
        if (rr < p.R) {
#pragma unroll
            for (int q = 0; q < 3; ++q) merge_any<kRes>(part, scratch[q * kM + m]);
            p.parts[(size_t)rr * p.P + cidx] = part;
            __threadfence();
        }
    }
    __syncthreads();
    const int grp = cidx / kGroup;
    const int gsize = min(kGroup, p.P - grp * kGroup);
    int* gcnt = p.gcount + blk * kMaxGroups + grp;
    if (threadIdx.x == 0) {
        if (aborted) {
            report(p.dev_status, DSPARK_ERR_TIMEOUT);
        } else {
            __threadfence();
            bar.last = (atomicAdd(gcnt, 1) == gsize - 1);
        }
    }
    __syncthreads();
    if (!bar.last) return;
    __threadfence();

    // ------------------------------------------- last CTA of its group: merge the group
    const int rows = min(kM, p.R - row0);
    TcPartial* stage = reinterpret_cast<TcPartial*>(sB);
    stage_partials(stage, p.parts + (size_t)row0 * p.P, p.P, grp * kGroup, gsize, rows);
    __syncthreads();
    for (int m = threadIdx.x; m < rows; m += kThreads) {
        TcPartial w = identity_partial<kRes>();
        for (int j = 0; j < gsize; ++j) merge_any<kRes>(w, stage[m * gsize + j]);
        p.gparts[(size_t)(row0 + m) * kMaxGroups + grp] = w;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        *gcnt = 0;  // ready for the next launch
        bar.top = (atomicAdd(p.tcount + blk, 1) == p.n_groups - 1);
    }
    __syncthreads();
    if (!bar.top) return;
    __threadfence();

    // ------------------------------------------- last group of the block: final merge
    stage_partials(stage, p.gparts + (size_t)row0 * kMaxGroups, kMaxGroups, 0, p.n_groups, rows);
    __syncthreads();
    for (int m = threadIdx.x; m < rows; m += kThreads) {
        const int rr = row0 + m;
        TcPartial w = identity_partial<kRes>();
        for (int j = 0; j < p.n_groups; ++j) merge_any<kRes>(w, stage[m * p.n_groups + j]);
        if (kRes) {
            const ResRow ri = p.rows[rr];
            if (ri.mode == 0) continue;
            const int alt = __float_as_int(w.m);
            int tok = (ri.mode == 1 && w.sum > 0.0f) ? w.idx : alt;
            if (tok < 0 || tok >= p.V) {  // no finite score (NaN logits)
                tok = -1;
                report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
            }
            p.out_tokens[(size_t)rr * (p.gamma + 1) + ri.pos] = tok;
        } else {
            const size_t rk = (size_t)rr * p.gamma + p.k;
            const int prev = prev_of(p, rr);
            if (prev == -2 || w.idx < 0 || w.idx >= p.V) {
                p.y[rk] = -1;
                if (p.q_lse) p.q_lse[rk] = NAN;
                if (p.q_tok) p.q_tok[rk] = NAN;
                report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
            } else {
                p.y[rk] = w.idx;
                if (!p.greedy) {
                    const float lse = w.m + logf(w.sum);
                    if (p.q_lse) p.q_lse[rk] = lse;
                    if (p.q_tok) p.q_tok[rk] = expf(w.s_at - lse);
                }
            }
        }
    }
    if (threadIdx.x == 0) p.tcount[blk] = 0;
    if (!kRes && p.k + 1 < p.gamma) {
        // the next step's A rows: H[r] = W1[y_k[r]] (zeros for an unusable request)
        __syncthreads();
        const int cpr = p.rank >> 3;
        const int total = rows * cpr;
        for (int e0 = threadIdx.x; e0 < total; e0 += 8 * kThreads) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * kThreads;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (e < total) {
                    const int m = e / cpr, c = e - m * cpr;
                    const int tok = p.y[(size_t)(row0 + m) * p.gamma + p.k];
                    if (tok >= 0 && tok < p.V) v[u] = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)tok * p.rank) + c);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * kThreads;
                if (e < total) {
                    const int m = e / cpr, c = e - m * cpr;
                    reinterpret_cast<uint4*>(p.H + (size_t)(row0 + m) * p.rank)[c] = v[u];
                }
            }
        }
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

struct TcLayout {
    size_t counters, parts, gparts, h, rows, total;
};
TcLayout tc_layout(int R, int rank, bool residual) {
    const int nb = (R + kM - 1) / kM;
    TcLayout L;
    size_t off = 0;
    L.counters = off; off += up256(sizeof(int) * (size_t)nb * (kMaxGroups + 1));
    L.parts = off; off += up256(sizeof(TcPartial) * (size_t)R * kMaxP);
    L.gparts = off; off += up256(sizeof(TcPartial) * (size_t)R * kMaxGroups);
    L.h = off; off += up256((size_t)R * rank * 2);
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
            void* ws, bool residual, TcParams& p, CUtensorMap& tm_w2, CUtensorMap& tm_u, CUtensorMap& tm_h,
            int& grid, size_t& smem, int& n_sm) {
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
    // the end-of-launch partial exchange and merges reuse the drained stages
    if ((size_t)n_stages * kTileBytes < (size_t)kM * kMaxGroups * sizeof(TcPartial)) return DSPARK_ERR_UNSUPPORTED;

    const TcLayout L = tc_layout(R, rank, residual);
    unsigned char* w = static_cast<unsigned char*>(ws);
    uint16_t* H = reinterpret_cast<uint16_t*>(w + L.h);
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
    p.H = H;
    p.parts = reinterpret_cast<TcPartial*>(w + L.parts);
    p.gparts = reinterpret_cast<TcPartial*>(w + L.gparts);
    p.R = R;
    p.gamma = gamma;
    p.V = V;
    p.rank = rank;
    p.nb = (R + kM - 1) / kM;
    p.gcount = reinterpret_cast<int*>(w + L.counters);
    p.tcount = p.gcount + (size_t)p.nb * kMaxGroups;
    p.n_tiles = (V + kNV - 1) / kNV;
    p.P = std::max(1, std::min(std::min(n_sm / p.nb, p.n_tiles), kMaxP));
    p.n_groups = (p.P + kGroup - 1) / kGroup;
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

size_t draft_tc_workspace(int R, int, int rank) { return tc_layout(R, rank, false).total; }

size_t residual_tc_workspace(int R, int rank) { return tc_layout(R, rank, true).total; }

int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    if (a.q_logits && (reinterpret_cast<uintptr_t>(a.q_logits) & 15)) return DSPARK_ERR_UNSUPPORTED;
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_h;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st = prepare(enc, a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, a.ws, false, p, tm_w2, tm_u, tm_h, grid,
                           smem, n_sm);
    if (st != DSPARK_OK) return st;
    p.anchor = a.anchor;
    p.seeds = a.seeds;
    p.y = a.y;
    p.q_lse = a.q_lse;
    p.q_tok = a.q_tok;
    p.q_logits = a.q_logits;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = a.greedy;
    if (cudaFuncSetAttribute(markov_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(p.gcount, 0, sizeof(int) * (size_t)p.nb * (kMaxGroups + 1), stream) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    {
        const long long chunks = (long long)a.R * (a.rank >> 3);
        const int blocks = (int)std::min<long long>((chunks + 255) / 256, 4LL * n_sm);
        gather_anchor_rows_kernel<<<blocks, 256, 0, stream>>>(p.W1, a.anchor, a.R, a.V, a.rank, p.H);
    }
    // Each step may start while the previous one finishes its reduction: the
    // kernel prefetches its first tiles and waits (griddepcontrol) before it
    // reads anything the previous launch wrote.
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
    for (int k = 0; k < a.gamma; ++k) {
        p.k = k;
        if (cudaLaunchKernelEx(&cfg, markov_tc_kernel<false>, tm_w2, tm_u, tm_h, p) != cudaSuccess)
            return DSPARK_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int launch_residual_tc(const ResidualTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    TcParams p;
    CUtensorMap tm_w2, tm_u, tm_h;
    int grid = 0, n_sm = 0;
    size_t smem = 0;
    const int st = prepare(enc, a.U, a.W1, a.W2, a.R, a.gamma, a.V, a.rank, a.ws, true, p, tm_w2, tm_u, tm_h, grid,
                           smem, n_sm);
    if (st != DSPARK_OK) return st;
    const TcLayout L = tc_layout(a.R, a.rank, true);
    ResRow* rows = reinterpret_cast<ResRow*>(static_cast<unsigned char*>(a.ws) + L.rows);
    p.anchor = a.anchor;
    p.y = const_cast<int32_t*>(a.y);
    p.seeds = a.seeds;
    p.dev_status = a.dev_status;
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = 0;
    p.target = a.target;
    p.rows = rows;
    p.out_tokens = a.out_tokens;
    if (cudaFuncSetAttribute(markov_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(p.gcount, 0, sizeof(int) * (size_t)p.nb * (kMaxGroups + 1), stream) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    {
        const long long chunks = (long long)a.R * (a.rank >> 3);
        const int blocks = (int)std::min<long long>((chunks + 255) / 256, 4LL * n_sm);
        residual_prep_kernel<<<blocks, 256, 0, stream>>>(a, rows, p.H);
    }
    p.k = 0;
    markov_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tm_w2, tm_u, tm_h, p);
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark

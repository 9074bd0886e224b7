// draft_tc.cu -- Markov-head draft step on the tcgen05 tensor cores.
//
// "DSpark explainer" (papers.franksyz.com topic 31) sections 6-7 and llama.cpp
// PR 25173 (draft-dspark): per block position k the drafter's logits are
// U_k + W2 . W1[prev] with prev the anchor (k = 0) or the token drafted at
// k - 1, sampled left to right; the PR's "future work" asks for the bias and
// the argmax fused into one kernel, which is what one launch here is.
//
// One launch per position k, persistent, one CTA per SM:
//   A (M = 128 requests x K = rank) = W1[prev] rows, gathered by the epilogue
//     warps into shared memory in the 128-byte-swizzled K-major layout and kept
//     resident for the whole launch;
//   B (N = 128 vocabulary rows x K = rank) = W2 tiles streamed by TMA through a
//     ring of 16 KB stages (64 rank elements per stage);
//   D = A . B^T accumulated in fp32 in tensor memory, two 128-column buffers so
//     the epilogue of one vocabulary tile overlaps the MMAs of the next;
//   epilogue (16 warps; thread = one request x 32 vocabulary columns, in two
//     16-column passes): adds the base logits U (prefetched into L2 by TMA and
//     read straight into registers), scales by 1/T, keeps (max, sum of exp) and
//     draws the Gumbel-max sample in its exponential-race form: with
//     w = exp(s - m) and E = -log(u), the largest s + Gumbel(u) = s - log(E) is
//     the largest w / E, so a candidate replaces the best when
//     w * E_best > w_best * E (one log and one exp per entry); optionally
//     stores the scaled logits q_logits.
// Each CTA leaves one partial per request; the last CTA to finish (atomic
// counter, no spin) reduces them, one warp per request, into y, q_lse, q_tok.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2-17 = gather + epilogue.  Every mbarrier wait is bounded (2 s); a
// timeout aborts the CTA cleanly and reports DSPARK_ERR_TIMEOUT.
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
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;

struct TcPartial {
    float score;
    int idx;
    float s_at;
    float m, sum;
    float pad[3];
};

struct TcParams {
    const uint16_t* U;
    const uint16_t* W1;
    const int32_t* anchor;
    const uint64_t* seeds;
    int32_t* y;
    float* q_lse;
    float* q_tok;
    float* q_logits;
    int32_t* dev_status;
    int* counter;
    TcPartial* parts;
    uint32_t cycle;
    float invT;
    int greedy;
    int R, gamma, V, rank, k;
    int nb, P, n_tiles, n_stages, nkb;
};

struct Bars {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t tfull[2], tempty[2];
    uint64_t afull, mma_done;
    uint32_t tmem_slot;
    int abort_flag;
    int last;
    int pad;
};

__device__ __forceinline__ void merge_partial(float& sc, int& ix, float& sa, float& m, float& su,
                                              float sc2, int ix2, float sa2, float m2, float su2) {
    if (better(sc2, ix2, sc, ix)) { sc = sc2; ix = ix2; sa = sa2; }
    lse_merge(m, su, m2, su2);
}

__device__ __forceinline__ int prev_of(const TcParams& p, int r) {  // -1 none, -2 bad
    if (p.k == 0) {
        const int a = p.anchor[r];
        return a >= p.V ? -2 : (a < 0 ? -1 : a);
    }
    const int t = p.y[(size_t)r * p.gamma + p.k - 1];
    return (t < 0 || t >= p.V) ? -2 : t;
}

__global__ void __launch_bounds__(kThreads, 1)
draft_step_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
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
        bar.last = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bar.tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tm_w2);
        tc::prefetch_tmap(&tm_u);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = bar.tmem_slot;
    const int n_local = cidx < p.n_tiles ? (p.n_tiles - 1 - cidx) / p.P + 1 : 0;

    // per-request running partial of this thread (epilogue threads)
    float best = -INFINITY, s_at = 0.0f, mx = -INFINITY, sum = 0.0f;
    int bidx = INT_MAX;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int last_phase[kMaxStages];
            for (int i = 0; i < kMaxStages; ++i) last_phase[i] = -1;
            bool ok = true;
            for (int i = 0; ok && i < n_local; ++i) {
                const int t = cidx + i * p.P;
                // base logits of this tile go to L2 while its W2 tile streams in
                tc::tma_prefetch_l2_3d(&tm_u, t * kNV, p.k, row0);
                tc::tma_prefetch_l2_3d(&tm_u, t * kNV + kKB, p.k, row0);
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!tc::mbar_wait(&bar.empty[s], ph ^ 1u, abort_flag, kWaitNs)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(&bar.full[s], kTileBytes);
                    tc::tma_load_2d(sB + s * kTileBytes, &tm_w2, &bar.full[s], kb * kKB, t * kNV);
                    last_phase[s] = (int)ph;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (*abort_flag) {
                // let the copies already in flight land before the CTA exits
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
        // ------------------------------------------------------------ gather + epilogue
        const int ew = warp - 2;           // 0..15
        const int quad = warp & 3;         // TMEM lane quadrant this warp may read
        const int quarter = ew >> 2;       // which 32 of the tile's 128 columns
        const int m = quad * 32 + lane;
        const int rr = row0 + m;
        {
            // A = W1[prev] rows, 16-byte chunks, eight loads in flight per thread
            const int cpr = p.rank >> 3;
            const int total = kM * cpr;
            const int et = threadIdx.x - 64;
            for (int base = 0; base < total; base += 8 * kEpiWarps * 32) {
                uint4 val[8];
                int dst_off[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = base + et + u * kEpiWarps * 32;
                    val[u] = make_uint4(0u, 0u, 0u, 0u);
                    dst_off[u] = -1;
                    if (e < total) {
                        const int row = e / cpr, c = e - row * cpr;
                        const int g = row0 + row;
                        const int prev = g < p.R ? prev_of(p, g) : -1;
                        if (prev >= 0) val[u] = __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)prev * p.rank) + c);
                        const int kb = c >> 3, cc = c & 7;
                        dst_off[u] = kb * kTileBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((cc ^ (row & 7)) << 4);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (dst_off[u] >= 0) *reinterpret_cast<uint4*>(sA + dst_off[u]) = val[u];
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar.afull);
        }
        const bool row_ok = rr < p.R;
        PhiloxKey K;
        if (!p.greedy) K = philox_key(row_ok ? p.seeds[rr] : 0ull);
        const uint32_t w3 = ctr_word3(p.cycle, kDraftGumbel);
        const size_t rk = (size_t)rr * p.gamma + p.k;
        const uint16_t* urow = p.U + rk * p.V;
        float* qrow = (p.q_logits && row_ok) ? p.q_logits + rk * p.V : nullptr;
        // exponential race state: best candidate's w (relative to mx) and E
        float bw = 0.0f, bE = 1.0f;
        for (int i = 0; i < n_local; ++i) {
            const int t = cidx + i * p.P;
            const int a = i & 1;
            const uint32_t use = (uint32_t)(i >> 1);
            const int vq = t * kNV + quarter * kCols;
            // base logits of this thread's 32 columns (already in L2), two halves
            uint32_t uwA[8], uwB[8];
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
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t word = h ? uwB[c >> 1] : uwA[c >> 1];
                    const float u = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
                    const float sb = u + sv[c];
                    sv[c] = p.greedy ? sb : sb * p.invT;
                }
                if (qrow) {
#pragma unroll
                    for (int c = 0; c < 16; c += 4)
                        if (c < nvalid)
                            *reinterpret_cast<float4*>(qrow + v0 + c) = make_float4(sv[c], sv[c + 1], sv[c + 2], sv[c + 3]);
                }
                if (p.greedy) {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c < nvalid && better(sv[c], v0 + c, best, bidx)) { best = sv[c]; bidx = v0 + c; s_at = sv[c]; }
                } else {
                    float cm = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 16; ++c) if (c < nvalid) cm = fmaxf(cm, sv[c]);
                    if (cm > mx) {
                        const float sc = expf(mx - cm);  // 0 while mx = -inf
                        sum *= sc;
                        bw *= sc;
                        mx = cm;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 wd = philox4x32_10(
                            make_uint4((uint32_t)((v0 >> 2) + q), (uint32_t)p.k, (uint32_t)rr, w3), K);
                        const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * q + e;
                            if (c < nvalid) {
                                const float w = expf(sv[c] - mx);
                                sum += w;
                                const float E = -logf(uniform_from_bits(words[e]));
                                if (w * bE > bw * E) { bw = w; bE = E; bidx = v0 + c; s_at = sv[c]; }
                            }
                        }
                    }
                }
            }
        }
        // the winner's Gumbel score s - log(E), for merging across threads and CTAs
        if (!p.greedy && bidx != INT_MAX) best = s_at - logf(bE);
    }

    // ---------------------------------------------------------------- per-CTA partials
    __syncthreads();
    TcPartial* scratch = reinterpret_cast<TcPartial*>(sB);  // W2 stages are drained
    if (warp >= 6) {
        const int m = (warp & 3) * 32 + lane;
        const int qtr = (warp - 2) >> 2;  // 1..3
        TcPartial& o = scratch[(qtr - 1) * kM + m];
        o.score = best; o.idx = bidx; o.s_at = s_at; o.m = mx; o.sum = sum;
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
            for (int q = 0; q < 3; ++q) {
                const TcPartial o = scratch[q * kM + m];
                merge_partial(best, bidx, s_at, mx, sum, o.score, o.idx, o.s_at, o.m, o.sum);
            }
            TcPartial w;
            w.score = best; w.idx = bidx; w.s_at = s_at; w.m = mx; w.sum = sum;
            w.pad[0] = w.pad[1] = w.pad[2] = 0.0f;
            p.parts[(size_t)rr * p.P + cidx] = w;
            __threadfence();
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (aborted) {
            report(p.dev_status, DSPARK_ERR_TIMEOUT);
        } else {
            __threadfence();
            bar.last = (atomicAdd(p.counter, 1) == (int)gridDim.x - 1);
        }
    }
    __syncthreads();
    if (!bar.last) return;
    __threadfence();

    // ---------------------------------------------------------------- last CTA: reduce
    for (int rr = warp; rr < p.R; rr += kThreads / 32) {
        float sc = -INFINITY, sa = 0.0f, m2 = -INFINITY, su = 0.0f;
        int ix = INT_MAX;
        const TcPartial* pr = p.parts + (size_t)rr * p.P;
        for (int j = lane; j < p.P; j += 32) {
            const float4 a4 = __ldcg(reinterpret_cast<const float4*>(pr + j));
            const float b0 = __ldcg(&pr[j].sum);
            merge_partial(sc, ix, sa, m2, su, a4.x, __float_as_int(a4.y), a4.z, a4.w, b0);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float sc2 = shfl_xor(sc, o), sa2 = shfl_xor(sa, o), mm2 = shfl_xor(m2, o), su2 = shfl_xor(su, o);
            const int ix2 = shfl_xor(ix, o);
            merge_partial(sc, ix, sa, m2, su, sc2, ix2, sa2, mm2, su2);
        }
        if (lane == 0) {
            const size_t rk = (size_t)rr * p.gamma + p.k;
            const int prev = prev_of(p, rr);
            if (prev == -2 || ix < 0 || ix >= p.V) {
                p.y[rk] = -1;
                if (p.q_lse) p.q_lse[rk] = NAN;
                if (p.q_tok) p.q_tok[rk] = NAN;
                report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
            } else {
                p.y[rk] = ix;
                if (!p.greedy) {
                    const float lse = m2 + logf(su);
                    if (p.q_lse) p.q_lse[rk] = lse;
                    if (p.q_tok) p.q_tok[rk] = expf(sa - lse);
                }
            }
        }
    }
    if (threadIdx.x == 0) *p.counter = 0;
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

struct TcLayout {
    size_t counter, parts, total;
};
TcLayout tc_layout(int R) {
    TcLayout L;
    size_t off = 0;
    L.counter = off; off += 256;
    L.parts = off; off += ((sizeof(TcPartial) * (size_t)R * kMaxP + 255) / 256) * 256;
    L.total = off;
    return L;
}

}  // namespace

bool draft_tc_supported(int u_dtype, int w_dtype, int R, int V, int rank) {
    return u_dtype == DSPARK_BF16 && w_dtype == DSPARK_BF16 && R >= 1 && rank % kKB == 0 && rank >= kKB &&
           rank <= 512 && V % 8 == 0 && V >= 8;
}

size_t draft_tc_workspace(int R, int, int) { return tc_layout(R).total; }

int launch_draft_tc(const DraftTcArgs& a, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return DSPARK_ERR_CUDA;
    if (a.q_logits && (reinterpret_cast<uintptr_t>(a.q_logits) & 15)) return DSPARK_ERR_UNSUPPORTED;
    int dev = 0, n_sm = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return DSPARK_ERR_CUDA;

    const int nkb = a.rank / kKB;
    const size_t fixed = 1024 + (size_t)nkb * kTileBytes + sizeof(Bars);
    if ((size_t)max_smem < fixed + 2 * kTileBytes) return DSPARK_ERR_UNSUPPORTED;
    const int n_stages = (int)std::min<size_t>(kMaxStages, ((size_t)max_smem - fixed) / kTileBytes);
    const size_t smem = fixed + (size_t)n_stages * kTileBytes;
    // the end-of-launch partial exchange reuses the drained stages
    if ((size_t)n_stages * kTileBytes < 3 * kM * sizeof(TcPartial)) return DSPARK_ERR_UNSUPPORTED;

    CUtensorMap tm_w2, tm_u;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.rank, (cuuint64_t)a.V};
        const cuuint64_t strides[1] = {(cuuint64_t)a.rank * 2};
        const cuuint32_t box[2] = {kKB, kNV};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_CUDA;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)a.V, (cuuint64_t)a.gamma, (cuuint64_t)a.R};
        const cuuint64_t strides[2] = {(cuuint64_t)a.V * 2, (cuuint64_t)a.gamma * a.V * 2};
        const cuuint32_t box[3] = {kKB, 1, kM};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tm_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.U), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_CUDA;
    }

    const TcLayout L = tc_layout(a.R);
    TcParams p;
    p.U = static_cast<const uint16_t*>(a.U);
    p.W1 = static_cast<const uint16_t*>(a.W1);
    p.anchor = a.anchor;
    p.seeds = a.seeds;
    p.y = a.y;
    p.q_lse = a.q_lse;
    p.q_tok = a.q_tok;
    p.q_logits = a.q_logits;
    p.dev_status = a.dev_status;
    p.counter = reinterpret_cast<int*>(static_cast<unsigned char*>(a.ws) + L.counter);
    p.parts = reinterpret_cast<TcPartial*>(static_cast<unsigned char*>(a.ws) + L.parts);
    p.cycle = a.cycle;
    p.invT = a.invT;
    p.greedy = a.greedy;
    p.R = a.R;
    p.gamma = a.gamma;
    p.V = a.V;
    p.rank = a.rank;
    p.nb = (a.R + kM - 1) / kM;
    p.n_tiles = (a.V + kNV - 1) / kNV;
    p.P = std::max(1, std::min(std::min(n_sm / p.nb, p.n_tiles), kMaxP));
    p.n_stages = n_stages;
    p.nkb = nkb;
    const int grid = p.P * p.nb;

    if (cudaFuncSetAttribute(draft_step_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(p.counter, 0, sizeof(int), stream) != cudaSuccess) return DSPARK_ERR_CUDA;
    for (int k = 0; k < a.gamma; ++k) {
        p.k = k;
        draft_step_tc_kernel<<<grid, kThreads, smem, stream>>>(tm_w2, tm_u, p);
    }
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark

// verify.cu -- lossless left-to-right verification of the drafted blocks.
//
// "DSpark explainer" (papers.franksyz.com topic 31) section 2: verify left to
// right, drop everything after the first rejection, emit a correction on
// rejection or a bonus token after full acceptance; section 3: accept with
// min(1, p/q), correct from max(0, p - q); section 13: the verified rows of
// all requests are packed back to back, delimited by cu_seqlens.
//
// Three launches:
//   verify_prologue  one CTA: checks cu_seqlens and the draft ids, clears the
//                    per-request counters, fills the outputs of bad requests;
//   verify_rounds    one cooperative launch, rounds j = 0, 1, ... over the
//                    block positions.  Round j streams row j of every request
//                    whose drafts 0..j-1 were all accepted: every warp walks
//                    its own sequence of 1024-element units with the next
//                    unit's loads in flight while it reduces the current one
//                    (max, sum of exp, first argmax of t = row * invT); after
//                    a grid barrier one warp per such request merges its units
//                    and decides draft j (or, at j = l, takes the bonus row);
//                    accepted requests go on to round j + 1 (published by a
//                    second grid barrier; when at most 16 requests are active,
//                    every CTA decides all of them itself instead and only the
//                    owner of a request writes its outputs).  Rows after the
//                    first rejection are never read: with a weak drafter a
//                    request needs about one row, with a strong one every
//                    round still streams at the full rate of the grid.
//   verify_correct   (T > 0) one CTA per (request, chunk) of the row the extra
//                    token comes from: Gumbel-max over log max(0, p - q) or
//                    over p; the last CTA of the request writes the token.
#include <algorithm>

#include "kernels.cuh"

namespace dspark {
namespace {

__global__ void __launch_bounds__(1024) verify_prologue_kernel(VerifyParams p) {
    __shared__ int bad_cu;
    if (threadIdx.x == 0) bad_cu = 0;
    __syncthreads();
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        const int a = p.cu[r], b = p.cu[r + 1];
        const int l = b - a - 1;
        if ((r == 0 && a != 0) || l < 0 || l > p.gamma || b > p.max_rows) atomicOr(&bad_cu, 1);
    }
    __syncthreads();
    const int ok = !bad_cu;
    if (threadIdx.x < 8) p.lazy[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        p.ok[0] = ok;
        if (!ok) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
        if (p.res_keys) p.res_keys[p.R] = 0ull;  // the residual launch's count of CTAs done
    }
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        p.cnt1[r] = 0;
        p.cnt2[r] = 0;
        int valid = ok;
        if (ok) {
            const int l = p.cu[r + 1] - p.cu[r] - 1;  // 0 <= l <= gamma <= 16 here
#pragma unroll
            for (int j = 0; j < 16; ++j) {  // independent loads, all in flight
                if (j < l) {
                    const int yj = p.y[(size_t)r * p.gamma + j];
                    if (yj < 0 || yj >= p.V) valid = 0;
                }
            }
            if (!valid) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
        }
        p.valid[r] = valid;
        VerifyJob job;  // no extra token until the request is decided
        job.row = 0; job.pos = 0; job.mode = 0; job.pad = 0; job.lse = 0.0f;
        job.pad2[0] = job.pad2[1] = job.pad2[2] = 0.0f;
        p.jobs[r] = job;
        p.act[r] = 0;
        p.act[p.R + r] = 0;
        if (p.res_rows) {  // nothing to draw until the request is decided
            ResRow w;
            w.mode = 0; w.pos = 0; w.trow = 0; w.w3 = 0; w.lse2_p = 0.0f; w.q_lse2 = 0.0f; w.prev = -1; w.pad = 0.0f;
            p.res_rows[r] = w;
            p.res_keys[r] = 0ull;
        }
        if (!valid) {
            p.n_acc[r] = -1;
            for (int j = 0; j <= p.gamma; ++j) p.out_tokens[(size_t)r * (p.gamma + 1) + j] = -1;
        }
    }
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// (max, sum of 2^(x - max)) pairs in base-2 units, merged.
__device__ __forceinline__ void lse2_merge(float& m, float& s, float m2, float s2) {
    if (m2 > m) {
        s = s * exp2f(m - m2) + s2;  // exp2f(-inf) = 0 covers an empty side
        m = m2;
    } else if (m2 != -INFINITY) {
        s = s + s2 * exp2f(m2 - m);
    }
}

// Greedy: running first argmax of the raw row.  Sampling: t2 = row * invT *
// log2(e), running (max, sum of 2^(t2 - max)); the argmax is not needed.
template <bool kGreedy>
__device__ __forceinline__ void stat_elem(float x, int v, float c2, float& m, float& s, float& bm, int& bi) {
    if (kGreedy) {
        if (x > bm) { bm = x; bi = v; }
    } else {
        const float t = x * c2;
        if (t > m) { s = s * exp2f(m - t) + 1.0f; m = t; }
        else s += exp2f(t - m);
    }
}

constexpr int kStatVec = kStatChunk / 4 / 32;  // float4 per lane and unit

// 16-byte loads of 1024-element piece `sub` of target row `row`,
// lane-interleaved (a warp reads 512 contiguous bytes per load); entries past
// the row end read as -inf and add nothing.
__device__ __forceinline__ void load_unit(const VerifyParams& p, int row, int sub, int lane, float4 (&b)[kStatVec]) {
    const int v0 = sub * kStatChunk, v1 = min(p.V, v0 + kStatChunk);
    const float* base = p.target + (size_t)row * p.V;
#pragma unroll
    for (int i = 0; i < kStatVec; ++i) {
        const int v = v0 + 4 * (lane + 32 * i);
        b[i] = v < v1 ? __ldcs(reinterpret_cast<const float4*>(base + v))
                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
}

// Round state in the workspace (zeroed by the prologue).
enum : int { kBarCount = 0, kBarGen = 1, kAbort = 2 };

// Grid-wide barrier of a cooperative launch (every CTA is resident): the last
// CTA to arrive resets the count and advances the generation; the others wait
// for it, at most p.wait_ns, after which the round state's abort flag is set.
// (p.phantom = 1 counts one arrival more than the grid has, so that nobody is
// last and every CTA's wait runs out: the timeout test.)  Returns false when
// the pass is aborted.
__device__ __forceinline__ bool grid_barrier(const VerifyParams& p, int* st, unsigned& gen) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const unsigned target = gen + 1;
        __threadfence();
        if (atomicAdd(reinterpret_cast<unsigned*>(st + kBarCount), 1u) == gridDim.x - 1u + (unsigned)p.phantom) {
            st[kBarCount] = 0;
            __threadfence();
            atomicExch(reinterpret_cast<unsigned*>(st + kBarGen), target);
        } else {
            const uint64_t t0 = global_ns();
            for (unsigned it = 1; *reinterpret_cast<volatile unsigned*>(st + kBarGen) != target; ++it) {
                if ((it & 31) == 0 &&
                    (*reinterpret_cast<volatile int*>(st + kAbort) || global_ns() - t0 > p.wait_ns)) {
                    atomicExch(st + kAbort, 1);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok && !*reinterpret_cast<volatile int*>(st + kAbort);
    }
    __syncthreads();
    gen += 1;
    return s_ok != 0;
}

// One CTA per SM, a grid barrier of n_sm arrivals.  16 warps of up to 128
// registers: with 24 warps the stream loop spilled at the 80-register cap and
// the verify call took 118.9 us at the R = 128 bench shape against 110.7 us
// here (20 warps: 114.0; 12: 112.1; 12 or 8 warps with two units in flight
// per warp instead of one: 114.6 and 125.7).
constexpr int kRoundThreads = 512;
constexpr int kRoundWarps = kRoundThreads / 32;
constexpr size_t kMaxListBytes = sizeof(int) * DSPARK_VERIFY_MAX_R;  // the round's request list in shared memory

// What the decision of request r at position j needs besides its row's
// statistics, fetched early so that it is in registers when they are merged.
struct DecideInputs {
    int r = -1, first = 0, l = 0, y = 0, valid = 0;
    float t = 0.0f, q = 1.0f;
    uint64_t seed = 0;
};

template <bool kGreedy>
__device__ __forceinline__ DecideInputs decide_inputs(const VerifyParams& p, int r, int j) {
    DecideInputs d;
    d.r = r;
    d.valid = p.valid[r];
    d.first = p.cu[r];
    d.l = p.cu[r + 1] - d.first - 1;
    if (d.valid && j < d.l && IN_BOUNDS(d.first + j < p.max_rows, p.dev_status)) {
        d.y = p.y[(size_t)r * p.gamma + j];
        if (!kGreedy) {
            d.t = __ldcg(p.target + (size_t)(d.first + j) * p.V + d.y);  // (the target may be host memory)
            d.q = p.q_tok[(size_t)r * p.gamma + j];
            d.seed = p.seeds[r];
        }
    }
    return d;
}

// One warp: merge request d.r's unit statistics of row j (stj, written by other
// CTAs in this launch: read from L2), decide draft j (or take the bonus row at
// j = l) and, when `write`, store the outputs.  Returns the number of accepted
// drafts once decided, -1 when draft j was accepted (the request goes on to
// round j + 1), -2 for a request with bad inputs.  Every lane returns the same.
template <bool kGreedy>
__device__ __forceinline__ int decide_request(const VerifyParams& p, const RowStat* stj, const DecideInputs& d,
                                              int j, float c2, bool write) {
    const int lane = threadIdx.x & 31;
    const int r = d.r, g = p.gamma;
    if (!d.valid) return -2;
    const RowStat* rs = stj + (size_t)r * p.nsub;
    float cm = -INFINITY, cs = 0.0f, am = -INFINITY;
    int ai = INT_MAX;
    // four statistics per lane in flight at a time
    for (int c0 = 0; c0 < p.nsub; c0 += 128) {
        float4 q4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = c0 + lane + 32 * i;
            q4[i] = c < p.nsub ? __ldcg(reinterpret_cast<const float4*>(rs + c))
                               : make_float4(-INFINITY, 0.0f, __int_as_float(INT_MAX), 0.0f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int qi = __float_as_int(q4[i].z);
            if (better(q4[i].x, qi, am, ai)) { am = q4[i].x; ai = qi; }
            if (!kGreedy) lse2_merge(cm, cs, q4[i].x, q4[i].y);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = shfl_xor(cm, o), s2 = shfl_xor(cs, o), am2 = shfl_xor(am, o);
        const int ai2 = shfl_xor(ai, o);
        lse2_merge(cm, cs, m2, s2);
        if (better(am2, ai2, am, ai)) { am = am2; ai = ai2; }
    }
    const float lse2 = kGreedy ? 0.0f : cm + log2f(cs);  // base-2 log-normaliser of row j
    int n = -1;  // the request's number of accepted drafts once decided
    if (j == d.l) {
        n = d.l;  // every draft accepted: the extra token comes from this row
    } else if (lane == 0) {
        bool accept;
        float pt;
        if (kGreedy) {
            accept = (d.y == ai);
            pt = accept ? 1.0f : 0.0f;
        } else {
            pt = exp2f(d.t * c2 - lse2);
            const float ratio = pt / d.q;
            const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)j, (uint32_t)r, ctr_word3(p.cycle, kAccept)),
                                          (uint32_t)(d.seed & 0xFFFFFFFFu), (uint32_t)(d.seed >> 32));
            accept = uniform_from_bits(w.x) < ratio;
        }
        if (write && p.p_tok) p.p_tok[(size_t)r * g + j] = pt;
        if (!accept) n = j;
    }
    n = __shfl_sync(0xFFFFFFFFu, n, 0);
    if (n < 0 || !write) return n;
    int32_t* out = p.out_tokens + (size_t)r * (g + 1);
    for (int jj = lane; jj <= g; jj += 32)
        if (jj != n) out[jj] = jj < n ? p.y[(size_t)r * g + jj] : -1;
    if (lane == 0) {
        p.n_acc[r] = n;
        if (kGreedy) {
            out[n] = (ai >= 0 && ai < p.V) ? ai : -1;
            if (out[n] < 0) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);  // NaN row
        } else {
            VerifyJob job;
            job.row = d.first + n;
            job.pos = n;
            job.mode = (n < d.l) ? 1 : 2;
            job.pad = 0;
            job.lse = lse2 * kLn2;  // natural log-normaliser of t = row * invT
            job.pad2[0] = job.pad2[1] = job.pad2[2] = 0.0f;
            p.jobs[r] = job;
            if (p.res_rows) {
                // the residual draw's row: a rejection at n draws from max(0, p - q) of
                // row n, whose drafter logits come from W1 of the token before
                // position n (the anchor at n = 0); full acceptance draws from p
                int prev = -1;
                if (job.mode == 1) {
                    prev = n == 0 ? p.anchor[r] : p.y[(size_t)r * g + n - 1];
                    if (prev >= p.V || prev < 0) prev = -1;
                }
                ResRow w;
                w.mode = job.mode;
                w.pos = n;
                w.trow = p.row_copy ? r : job.row;  // the residual reads the device copy of the row
                w.w3 = ctr_word3(p.cycle, job.mode == 1 ? kResidualGumbel : kBonusGumbel);
                w.lse2_p = lse2;
                w.q_lse2 = job.mode == 1 ? p.q_lse[(size_t)r * g + n] * kLog2e : 0.0f;
                w.prev = prev;
                w.pad = 0.0f;
                p.res_rows[r] = w;
                // the residual launch reads this W1 row first (its A row)
                if (prev >= 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.W1 + (size_t)prev * p.rank),
                                 "r"((uint32_t)p.rank * 2u)
                                 : "memory");
            }
        }
    }
    return n;
}

template <bool kGreedy>
__global__ void __launch_bounds__(kRoundThreads, 1) verify_rounds_kernel(VerifyParams p) {
    extern __shared__ int s_list[];  // [R] the requests active in the current round
    __shared__ int s_nact;
    __shared__ int s_next[kRoundWarps];
    if (!p.ok[0]) return;  // the same for every CTA
    const int V = p.V, g = p.gamma;
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const int w0 = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * (size_t)blockDim.x) >> 5);
    const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.target) & 15) == 0);
    const float c2 = p.invT * kLog2e;
    int* st = p.lazy;
    unsigned gen = 0;
    int n_act = p.R;           // round 0: every request (the bad ones are skipped when deciding)
    bool all = true;           // round 0: request a is a
    for (int j = 0; j <= g && n_act > 0; ++j) {
        auto act_at = [&](int a) { return all ? a : s_list[a]; };
        // statistics of round j: two buffers by round parity, so that a CTA
        // already streaming round j + 1 never overwrites what another CTA still
        // merges for round j
        RowStat* stj = p.stats + (size_t)(j & 1) * p.R * p.nsub;
        // Few active requests: every CTA decides all of them itself (one warp
        // each, the same result everywhere; outputs written by one owner CTA)
        // and needs no second grid barrier.  Otherwise one warp of the grid per
        // request decides, and a barrier publishes the accept flags.
        const bool local = n_act <= kRoundWarps;
        const int dw = local ? wl : w0;  // the warp that will decide active request dw
        // its decision inputs now, so they are in registers after the stream
        DecideInputs din;
        if (dw < n_act && lane == 0) din = decide_inputs<kGreedy>(p, act_at(dw), j);
        // ---- row j of every active request: unit statistics
        const int n_units = n_act * p.nsub;
        auto unit_row = [&](int u, int& r, int& sub) {
            const int a = u / p.nsub;
            sub = u - a * p.nsub;
            r = act_at(a);
            const int row = __ldg(p.cu + r) + j;
            // (a debug build: a row outside the packed target is read as row 0)
            return IN_BOUNDS(row >= 0 && row < p.max_rows && r >= 0 && r < p.R, p.dev_status) ? row : 0;
        };
        float4 buf[kStatVec];
        if (vec && w0 < n_units) {
            int r0, sub0;
            const int row0 = unit_row(w0, r0, sub0);
            load_unit(p, row0, sub0, lane, buf);
        }
        for (int u = w0; u < n_units; u += nw) {
            int r, sub;
            const int row = unit_row(u, r, sub);
            const int v0 = sub * kStatChunk;
            // the next unit's loads go out before this one is reduced
            float4 nxt[kStatVec];
            if (vec && u + nw < n_units) {
                int r1, sub1;
                const int row1 = unit_row(u + nw, r1, sub1);
                load_unit(p, row1, sub1, lane, nxt);
            }
            float m = -INFINITY, s = 0.0f, bm = -INFINITY;
            int bi = INT_MAX;
            if (vec && p.row_copy) {  // host-resident target: keep the request's latest row on the device
                float* dst = p.row_copy + (size_t)r * V;
#pragma unroll
                for (int i = 0; i < kStatVec; ++i) {
                    const int v = v0 + 4 * (lane + 32 * i);
                    if (v < V) *reinterpret_cast<float4*>(dst + v) = buf[i];
                }
            }
            if (vec) {
                if (kGreedy) {
#pragma unroll
                    for (int i = 0; i < kStatVec; ++i) {
                        const int v = v0 + 4 * (lane + 32 * i);
                        stat_elem<true>(buf[i].x, v + 0, c2, m, s, bm, bi);
                        stat_elem<true>(buf[i].y, v + 1, c2, m, s, bm, bi);
                        stat_elem<true>(buf[i].z, v + 2, c2, m, s, bm, bi);
                        stat_elem<true>(buf[i].w, v + 3, c2, m, s, bm, bi);
                    }
                } else {
                    // the lane's maximum first, then one pass of 2^(t - max)
#pragma unroll
                    for (int i = 0; i < kStatVec; ++i) {
                        buf[i].x *= c2; buf[i].y *= c2; buf[i].z *= c2; buf[i].w *= c2;
                        m = fmaxf(m, fmaxf(fmaxf(buf[i].x, buf[i].y), fmaxf(buf[i].z, buf[i].w)));
                    }
                    if (m != -INFINITY) {
#pragma unroll
                        for (int i = 0; i < kStatVec; ++i)
                            s += (exp2f(buf[i].x - m) + exp2f(buf[i].y - m)) + (exp2f(buf[i].z - m) + exp2f(buf[i].w - m));
                    }
                }
            } else {
                const int v1 = min(V, v0 + kStatChunk);
                const float* base = p.target + (size_t)row * V;
                for (int v = v0 + lane; v < v1; v += 32) {
                    const float x = __ldcg(base + v);
                    if (p.row_copy) p.row_copy[(size_t)r * V + v] = x;
                    stat_elem<kGreedy>(x, v, c2, m, s, bm, bi);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = shfl_xor(m, o), s2 = shfl_xor(s, o), bm2 = shfl_xor(bm, o);
                const int bi2 = shfl_xor(bi, o);
                lse2_merge(m, s, m2, s2);
                if (better(bm2, bi2, bm, bi)) { bm = bm2; bi = bi2; }
            }
            if (lane == 0) {
                RowStat stt;
                stt.m = kGreedy ? bm : m;
                stt.s = s;
                stt.idx = bi;
                stt.pad = 0;
                stj[(size_t)r * p.nsub + sub] = stt;
            }
#pragma unroll
            for (int i = 0; i < kStatVec; ++i) buf[i] = nxt[i];
        }
        if (!grid_barrier(p, st, gen)) break;
        // the decision inputs fetched by lane 0, for the whole warp
        din.r = __shfl_sync(0xFFFFFFFFu, din.r, 0);
        din.valid = __shfl_sync(0xFFFFFFFFu, din.valid, 0);
        din.first = __shfl_sync(0xFFFFFFFFu, din.first, 0);
        din.l = __shfl_sync(0xFFFFFFFFu, din.l, 0);
        if (local) {
            // ---- every CTA: warp a decides active request a; the owner CTA writes
            int nx = -1;
            if (wl < n_act) {
                const int r = din.r;
                const int n = decide_request<kGreedy>(p, stj, din, j, c2, r % (int)gridDim.x == (int)blockIdx.x);
                nx = n == -1 ? r : -1;
            }
            if (lane == 0) s_next[wl] = nx;
            __syncthreads();
            if (threadIdx.x < 32) {
                const int v = lane < n_act ? s_next[lane] : -1;  // n_act <= kRoundWarps <= 32
                const unsigned msk = __ballot_sync(0xFFFFFFFFu, v >= 0);
                if (v >= 0) s_list[__popc(msk & ((1u << lane) - 1u))] = v;
                if (lane == 0) s_nact = __popc(msk);
            }
            __syncthreads();
        } else {
            // ---- one warp of the grid per active request: decide draft j
            for (int a = w0; a < n_act; a += nw) {
                // a == w0 was fetched at the round start (lane 0)
                const DecideInputs d = (a == w0) ? din : decide_inputs<kGreedy>(p, act_at(a), j);
                const int n = decide_request<kGreedy>(p, stj, d, j, c2, true);
                if (n == -1 && lane == 0) p.act[d.r] = j + 1;  // goes on to round j + 1
            }
            if (!grid_barrier(p, st, gen)) break;
            // every CTA lists the requests accepted in this round (flags written by
            // other CTAs: read from L2)
            if (threadIdx.x < 32) {
                int cnt = 0;
                for (int base = 0; base < p.R; base += 32) {
                    const bool f = base + lane < p.R && __ldcg(p.act + base + lane) == j + 1;
                    const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
                    if (f) s_list[cnt + __popc(m & ((1u << lane) - 1u))] = base + lane;
                    cnt += __popc(m);
                }
                if (lane == 0) s_nact = cnt;
            }
            __syncthreads();
        }
        n_act = s_nact;
        all = false;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && *reinterpret_cast<volatile int*>(st + kAbort))
        report(p.dev_status, DSPARK_ERR_TIMEOUT);
}

__device__ __forceinline__ void block_sample(float& best, int& idx, float& best2, int& idx2,
                                             float& mass) {
    __shared__ float sb[32], sb2[32], sms[32];
    __shared__ int si[32], si2[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float b = shfl_xor(best, o), b2 = shfl_xor(best2, o), ms = shfl_xor(mass, o);
        const int i = shfl_xor(idx, o), i2 = shfl_xor(idx2, o);
        if (better(b, i, best, idx)) { best = b; idx = i; }
        if (better(b2, i2, best2, idx2)) { best2 = b2; idx2 = i2; }
        mass += ms;
    }
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sb[w] = best; si[w] = idx; sb2[w] = best2; si2[w] = idx2; sms[w] = mass; }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        best = lane < nw ? sb[lane] : -INFINITY;
        idx = lane < nw ? si[lane] : INT_MAX;
        best2 = lane < nw ? sb2[lane] : -INFINITY;
        idx2 = lane < nw ? si2[lane] : INT_MAX;
        mass = lane < nw ? sms[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float b = shfl_xor(best, o), b2 = shfl_xor(best2, o), ms = shfl_xor(mass, o);
            const int i = shfl_xor(idx, o), i2 = shfl_xor(idx2, o);
            if (better(b, i, best, idx)) { best = b; idx = i; }
            if (better(b2, i2, best2, idx2)) { best2 = b2; idx2 = i2; }
            mass += ms;
        }
    }
}

__global__ void __launch_bounds__(kVerifyThreads) verify_correct_kernel(VerifyParams p) {
    __shared__ int s_last;
    const int r = blockIdx.x / p.nchunk;
    const int chunk = blockIdx.x - r * p.nchunk;
    if (!p.ok[0] || !p.valid[r]) return;
    // a decision pass that gave up (a grid barrier's wait ran out) leaves
    // requests undecided: nothing to draw for them
    if (*reinterpret_cast<volatile int*>(p.lazy + kAbort)) return;
    const VerifyJob job = p.jobs[r];
    if (job.mode == 0) return;
    if (!IN_BOUNDS(job.row >= 0 && job.row < p.max_rows && job.pos >= 0 &&
                       (job.mode == 1 ? job.pos < p.gamma : job.pos <= p.gamma),  // a bonus draws at pos = l <= gamma
                   p.dev_status))
        return;
    const int V = p.V;
    const int v0 = chunk * kVerifyChunk;
    const int v1 = min(V, v0 + kVerifyChunk);
    const float* trow = p.target + (size_t)job.row * V;
    const int g = p.gamma;
    const bool residual = job.mode == 1;
    const float* qrow = residual ? p.q_logits + ((size_t)r * g + job.pos) * V : nullptr;
    const float qlse = residual ? p.q_lse[(size_t)r * g + job.pos] : 0.0f;
    const PhiloxKey K = philox_key(p.seeds[r]);
    const uint32_t w3 = ctr_word3(p.cycle, residual ? kResidualGumbel : kBonusGumbel);

    float best = -INFINITY, best2 = -INFINITY, mass = 0.0f;
    int idx = INT_MAX, idx2 = INT_MAX;
    // groups of 4 vocabulary entries share one Philox call (lane = v & 3)
    for (int v4 = (v0 >> 2) + threadIdx.x; 4 * v4 < v1; v4 += kVerifyThreads) {
        const uint4 wd = philox4x32_10(make_uint4((uint32_t)v4, (uint32_t)job.pos, (uint32_t)r, w3), K);
        const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = 4 * v4 + i;
            if (v >= v1) break;
            const float t = __ldg(trow + v) * p.invT;
            const float gn = gumbel_from_uniform(uniform_from_bits(words[i]));
            const float alt = t + gn;
            if (better(alt, v, best2, idx2)) { best2 = alt; idx2 = v; }
            if (residual) {
                const float pv = expf(t - job.lse);
                const float qv = expf(__ldg(qrow + v) - qlse);
                const float res = pv - qv;
                if (res > 0.0f) {
                    mass += res;
                    const float sc = logf(res) + gn;
                    if (better(sc, v, best, idx)) { best = sc; idx = v; }
                }
            }
        }
    }
    block_sample(best, idx, best2, idx2, mass);
    if (threadIdx.x == 0) {
        SamplePartial sp;
        sp.best = best; sp.idx = idx; sp.best_alt = best2; sp.idx_alt = idx2; sp.mass = mass;
        sp.pad[0] = sp.pad[1] = sp.pad[2] = 0.0f;
        p.parts[(size_t)r * p.nchunk + chunk] = sp;
        __threadfence();
        s_last = (atomicAdd(p.cnt2 + r, 1) == p.nchunk - 1);
    }
    __syncthreads();
    if (!s_last || threadIdx.x != 0) return;
    __threadfence();
    float fb = -INFINITY, fb2 = -INFINITY, fm = 0.0f;
    int fi = INT_MAX, fi2 = INT_MAX;
    for (int c = 0; c < p.nchunk; ++c) {
        const SamplePartial* q = p.parts + (size_t)r * p.nchunk + c;
        const float b = __ldcg(&q->best), b2 = __ldcg(&q->best_alt);
        const int i = __ldcg(&q->idx), i2 = __ldcg(&q->idx_alt);
        if (better(b, i, fb, fi)) { fb = b; fi = i; }
        if (better(b2, i2, fb2, fi2)) { fb2 = b2; fi2 = i2; }
        fm += __ldcg(&q->mass);
    }
    int tok = (residual && fm > 0.0f) ? fi : fi2;
    if (tok < 0 || tok >= V) {  // no finite score (NaN logits)
        tok = -1;
        report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
    }
    p.out_tokens[(size_t)r * (g + 1) + job.pos] = tok;
}

}  // namespace

cudaError_t launch_verify_decide(const VerifyParams& p, cudaStream_t stream) {
    verify_prologue_kernel<<<1, 1024, 0, stream>>>(p);
    int dev = 0, n_sm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaGetLastError();
    const void* fn = p.greedy ? reinterpret_cast<const void*>(verify_rounds_kernel<true>)
                              : reinterpret_cast<const void*>(verify_rounds_kernel<false>);
    if ((size_t)p.R * sizeof(int) > kMaxListBytes) return cudaErrorInvalidValue;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxListBytes) != cudaSuccess)
        return cudaGetLastError();
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRoundThreads, sizeof(int) * p.R);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    // every CTA resident at once (cooperative launch): the rounds meet at grid barriers.
    // One CTA per SM, but no more CTAs than round 0 has units for one per warp: a
    // small batch (R = 1, V = 64: one unit) meets at a barrier of one CTA instead of
    // one per SM.
    const long long units0 = (long long)p.R * p.nsub;
    const int grid = (int)std::min<long long>(n_sm, std::max<long long>(1, (units0 + kRoundWarps - 1) / kRoundWarps));
    const size_t smem = sizeof(int) * (size_t)p.R;
    VerifyParams arg = p;
    arg.wait_ns = grid_wait_limit_ns();
    arg.phantom = (fault_injection_mask() & DSPARK_INJECT_VERIFY_BARRIER) ? 1 : 0;
    void* args[] = {&arg};
    e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kRoundThreads), args, smem, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
    const cudaError_t e = launch_verify_decide(p, stream);
    if (e != cudaSuccess) return e;
    if (!p.greedy) {
        const long long grid2 = (long long)p.R * p.nchunk;
        verify_correct_kernel<<<(unsigned)grid2, kVerifyThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace dspark

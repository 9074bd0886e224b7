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
//   verify_stats     one CTA per (row, 8192-element chunk): a streaming pass
//                    computing max, sum of exp and the first argmax of
//                    t = row * invT.  The last CTA of a request (counter, no
//                    spin) combines its rows and makes the accept decisions;
//   verify_correct   (T > 0) one CTA per (request, chunk) of the row the extra
//                    token comes from: Gumbel-max over log max(0, p - q) or
//                    over p; the last CTA of the request writes the token.
#include "kernels.cuh"

namespace dspark {
namespace {

__device__ __forceinline__ int request_of_row(const int32_t* cu, int R, int row) {
    // largest r with cu[r] <= row (cu non-decreasing, checked by the prologue)
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

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
    if (threadIdx.x == 0) {
        p.ok[0] = ok;
        if (!ok) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
    }
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        p.cnt1[r] = 0;
        p.cnt2[r] = 0;
        int valid = ok;
        if (ok) {
            const int l = p.cu[r + 1] - p.cu[r] - 1;
            for (int j = 0; j < l; ++j) {
                const int yj = p.y[(size_t)r * p.gamma + j];
                if (yj < 0 || yj >= p.V) valid = 0;
            }
            if (!valid) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
        }
        p.valid[r] = valid;
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

// Block-wide combine of (m, s, argmax) held by every thread (m, s in base-2
// units); result in thread 0.
__device__ __forceinline__ void block_rowstat(float& m, float& s, float& bm, int& bi) {
    __shared__ float sm_m[32], sm_s[32], sm_bm[32];
    __shared__ int sm_bi[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = shfl_xor(m, o), s2 = shfl_xor(s, o), bm2 = shfl_xor(bm, o);
        const int bi2 = shfl_xor(bi, o);
        lse2_merge(m, s, m2, s2);
        if (better(bm2, bi2, bm, bi)) { bm = bm2; bi = bi2; }
    }
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sm_m[w] = m; sm_s[w] = s; sm_bm[w] = bm; sm_bi[w] = bi; }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        m = lane < nw ? sm_m[lane] : -INFINITY;
        s = lane < nw ? sm_s[lane] : 0.0f;
        bm = lane < nw ? sm_bm[lane] : -INFINITY;
        bi = lane < nw ? sm_bi[lane] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = shfl_xor(m, o), s2 = shfl_xor(s, o), bm2 = shfl_xor(bm, o);
            const int bi2 = shfl_xor(bi, o);
            lse2_merge(m, s, m2, s2);
            if (better(bm2, bi2, bm, bi)) { bm = bm2; bi = bi2; }
        }
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

template <bool kGreedy>
__global__ void __launch_bounds__(kVerifyThreads) verify_stats_kernel(VerifyParams p) {
    __shared__ int s_req, s_last;
    const int row = blockIdx.x / p.nchunk;
    const int chunk = blockIdx.x - row * p.nchunk;
    if (!p.ok[0]) return;
    const int n_rows = p.cu[p.R];
    if (row >= n_rows) return;
    if (threadIdx.x == 0) s_req = request_of_row(p.cu, p.R, row);
    __syncthreads();
    const int r = s_req;
    if (!p.valid[r]) return;

    const int V = p.V;
    const int v0 = chunk * kVerifyChunk;
    const int v1 = min(V, v0 + kVerifyChunk);
    const float* base = p.target + (size_t)row * V;
    const float c2 = p.invT * kLog2e;
    float m = -INFINITY, s = 0.0f, bm = -INFINITY;
    int bi = INT_MAX;
    if ((V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.target) & 15) == 0)) {
        // 8 independent 16-byte loads per thread, then the arithmetic
        constexpr int kVec = kVerifyChunk / 4 / kVerifyThreads;
        float4 buf[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            const int v = v0 + 4 * (threadIdx.x + i * kVerifyThreads);
            buf[i] = v < v1 ? __ldcs(reinterpret_cast<const float4*>(base + v))
                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        if (kGreedy) {
#pragma unroll
            for (int i = 0; i < kVec; ++i) {
                const int v = v0 + 4 * (threadIdx.x + i * kVerifyThreads);
                if (v < v1) {
                    stat_elem<true>(buf[i].x, v + 0, c2, m, s, bm, bi);
                    stat_elem<true>(buf[i].y, v + 1, c2, m, s, bm, bi);
                    stat_elem<true>(buf[i].z, v + 2, c2, m, s, bm, bi);
                    stat_elem<true>(buf[i].w, v + 3, c2, m, s, bm, bi);
                }
            }
        } else {
            // the thread's maximum first, then one pass of 2^(t - max); entries past
            // the row end were loaded as -inf and add nothing
#pragma unroll
            for (int i = 0; i < kVec; ++i) {
                buf[i].x *= c2; buf[i].y *= c2; buf[i].z *= c2; buf[i].w *= c2;
                m = fmaxf(m, fmaxf(fmaxf(buf[i].x, buf[i].y), fmaxf(buf[i].z, buf[i].w)));
            }
            if (m != -INFINITY) {
#pragma unroll
                for (int i = 0; i < kVec; ++i)
                    s += (exp2f(buf[i].x - m) + exp2f(buf[i].y - m)) + (exp2f(buf[i].z - m) + exp2f(buf[i].w - m));
            }
        }
    } else {
        for (int v = v0 + threadIdx.x; v < v1; v += kVerifyThreads)
            stat_elem<kGreedy>(__ldg(base + v), v, c2, m, s, bm, bi);
    }
    block_rowstat(m, s, bm, bi);
    if (threadIdx.x == 0) {
        RowStat st;
        st.m = kGreedy ? bm : m;
        st.s = s;
        st.idx = bi;
        st.pad = 0;
        p.stats[(size_t)row * p.nchunk + chunk] = st;
        __threadfence();
        const int total = (p.cu[r + 1] - p.cu[r]) * p.nchunk;
        s_last = (atomicAdd(p.cnt1 + r, 1) == total - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of request r: combine its rows, decide left to right ----
    __shared__ float row_lse[17];
    __shared__ int row_amax[17];
    const int first = p.cu[r];
    const int l = p.cu[r + 1] - first - 1;
    if (threadIdx.x <= l) {
        const RowStat* rs = p.stats + (size_t)(first + threadIdx.x) * p.nchunk;
        float cm = -INFINITY, cs = 0.0f, am = -INFINITY;
        int ai = INT_MAX;
        for (int c = 0; c < p.nchunk; ++c) {
            const float m2 = __ldcg(&rs[c].m), s2 = __ldcg(&rs[c].s);
            const int i2 = __ldcg(&rs[c].idx);
            if (better(m2, i2, am, ai)) { am = m2; ai = i2; }
            if (!kGreedy) lse2_merge(cm, cs, m2, s2);
        }
        row_lse[threadIdx.x] = kGreedy ? 0.0f : cm + log2f(cs);  // base-2 log-normaliser
        row_amax[threadIdx.x] = ai;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int g = p.gamma;
        int n = l;
        for (int j = 0; j < l; ++j) {
            const int yj = p.y[(size_t)r * g + j];
            bool accept;
            float pt;
            if (kGreedy) {
                accept = (yj == row_amax[j]);
                pt = accept ? 1.0f : 0.0f;
            } else {
                pt = exp2f(p.target[(size_t)(first + j) * p.V + yj] * c2 - row_lse[j]);
                const float ratio = pt / p.q_tok[(size_t)r * g + j];
                const uint4 w = philox4x32_10(
                    make_uint4(0u, (uint32_t)j, (uint32_t)r, ctr_word3(p.cycle, kAccept)),
                    (uint32_t)(p.seeds[r] & 0xFFFFFFFFu), (uint32_t)(p.seeds[r] >> 32));
                accept = uniform_from_bits(w.x) < ratio;
            }
            if (p.p_tok) p.p_tok[(size_t)r * g + j] = pt;
            if (!accept) { n = j; break; }
        }
        p.n_acc[r] = n;
        int32_t* out = p.out_tokens + (size_t)r * (g + 1);
        for (int j = 0; j < n; ++j) out[j] = p.y[(size_t)r * g + j];
        for (int j = n + 1; j <= g; ++j) out[j] = -1;
        if (kGreedy) {
            const int tok = row_amax[n];
            out[n] = (tok >= 0 && tok < p.V) ? tok : -1;
            if (out[n] < 0) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);  // NaN row
        } else {
            VerifyJob job;
            job.row = first + n;
            job.pos = n;
            job.mode = (n < l) ? 1 : 2;
            job.pad = 0;
            job.lse = row_lse[n] * kLn2;  // natural log-normaliser of t = row * invT
            job.pad2[0] = job.pad2[1] = job.pad2[2] = 0.0f;
            p.jobs[r] = job;
        }
    }
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
    const VerifyJob job = p.jobs[r];
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
    const long long grid1 = (long long)p.max_rows * p.nchunk;
    if (grid1 > 0) {
        if (p.greedy) verify_stats_kernel<true><<<(unsigned)grid1, kVerifyThreads, 0, stream>>>(p);
        else verify_stats_kernel<false><<<(unsigned)grid1, kVerifyThreads, 0, stream>>>(p);
    }
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

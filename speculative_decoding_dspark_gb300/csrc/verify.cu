// verify.cu -- lossless left-to-right verification of the drafted blocks.
//
// "DSpark explainer" (papers.franksyz.com topic 31) section 2: verify left to
// right, drop everything after the first rejection, emit a correction on
// rejection or a bonus token after full acceptance; section 3: accept with
// min(1, p/q), correct from max(0, p - q); section 13: the verified rows of
// all requests are packed back to back, delimited by cu_seqlens.
//
// Four launches:
//   verify_prologue  one CTA: checks cu_seqlens and the draft ids, clears the
//                    per-request counters, fills the outputs of bad requests;
//   verify_stats     a streaming pass over (row, 1024-element) units, every
//                    warp on its own sequence of units with the next one's
//                    loads in flight while it reduces the current one: max,
//                    sum of exp and the first argmax of t = row * invT per
//                    unit; no block barrier, fence or atomic in the stream;
//   verify_decide    one CTA per request: combines its rows' units and
//                    makes the accept decisions, one thread per position;
//   verify_correct   (T > 0) one CTA per (request, chunk) of the row the extra
//                    token comes from: Gumbel-max over log max(0, p - q) or
//                    over p; the last CTA of the request writes the token.
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
constexpr int kStatThreads = 256;

// 16-byte loads of unit u = (row, 1024-element piece) of the packed target
// rows, lane-interleaved (a warp reads 512 contiguous bytes per load); entries
// past the row end read as -inf and add nothing.
__device__ __forceinline__ void load_unit(const VerifyParams& p, int u, int lane, float4 (&b)[kStatVec]) {
    const int row = u / p.nsub, sub = u - row * p.nsub;
    const int v0 = sub * kStatChunk, v1 = min(p.V, v0 + kStatChunk);
    const float* base = p.target + (size_t)row * p.V;
#pragma unroll
    for (int i = 0; i < kStatVec; ++i) {
        const int v = v0 + 4 * (lane + 32 * i);
        b[i] = v < v1 ? __ldcs(reinterpret_cast<const float4*>(base + v))
                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
}

template <bool kGreedy>
__global__ void __launch_bounds__(kStatThreads) verify_stats_kernel(VerifyParams p) {
    if (!p.ok[0]) return;
    const int V = p.V;
    const int n_units = p.cu[p.R] * p.nsub;
    const int lane = threadIdx.x & 31;
    const int w0 = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * (size_t)blockDim.x) >> 5);
    const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.target) & 15) == 0);
    const float c2 = p.invT * kLog2e;
    float4 buf[kStatVec];
    if (vec && w0 < n_units) load_unit(p, w0, lane, buf);
    for (int u = w0; u < n_units; u += nw) {
        const int row = u / p.nsub;
        const int sub = u - row * p.nsub;
        const int v0 = sub * kStatChunk;
        // the next unit's loads go out before this one is reduced
        float4 nxt[kStatVec];
        if (vec && u + nw < n_units) load_unit(p, u + nw, lane, nxt);
        float m = -INFINITY, s = 0.0f, bm = -INFINITY;
        int bi = INT_MAX;
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
            for (int v = v0 + lane; v < v1; v += 32) stat_elem<kGreedy>(__ldg(base + v), v, c2, m, s, bm, bi);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = shfl_xor(m, o), s2 = shfl_xor(s, o), bm2 = shfl_xor(bm, o);
            const int bi2 = shfl_xor(bi, o);
            lse2_merge(m, s, m2, s2);
            if (better(bm2, bi2, bm, bi)) { bm = bm2; bi = bi2; }
        }
        if (lane == 0) {
            RowStat st;
            st.m = kGreedy ? bm : m;
            st.s = s;
            st.idx = bi;
            st.pad = 0;
            p.stats[(size_t)row * p.nsub + sub] = st;
        }
#pragma unroll
        for (int i = 0; i < kStatVec; ++i) buf[i] = nxt[i];
    }
}

// One CTA per request: each row's units combined by a warp, then the drafts
// decided left to right (one thread per position; the first rejection wins).
template <bool kGreedy>
__global__ void __launch_bounds__(kStatThreads) verify_decide_kernel(VerifyParams p) {
    __shared__ float row_lse[17];
    __shared__ int row_amax[17];
    __shared__ float s_pt[16];
    __shared__ int s_acc[16];
    const int r = blockIdx.x;
    if (!p.ok[0] || !p.valid[r]) return;
    const int first = p.cu[r];
    const int l = p.cu[r + 1] - first - 1;
    const int g = p.gamma;
    const float c2 = p.invT * kLog2e;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j <= l; j += kStatThreads / 32) {
        const RowStat* rs = p.stats + (size_t)(first + j) * p.nsub;
        float cm = -INFINITY, cs = 0.0f, am = -INFINITY;
        int ai = INT_MAX;
        for (int c = lane; c < p.nsub; c += 32) {
            const RowStat q = rs[c];
            if (better(q.m, q.idx, am, ai)) { am = q.m; ai = q.idx; }
            if (!kGreedy) lse2_merge(cm, cs, q.m, q.s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = shfl_xor(cm, o), s2 = shfl_xor(cs, o), am2 = shfl_xor(am, o);
            const int ai2 = shfl_xor(ai, o);
            lse2_merge(cm, cs, m2, s2);
            if (better(am2, ai2, am, ai)) { am = am2; ai = ai2; }
        }
        if (lane == 0) {
            row_lse[j] = kGreedy ? 0.0f : cm + log2f(cs);  // base-2 log-normaliser
            row_amax[j] = ai;
        }
    }
    __syncthreads();
    const int j = threadIdx.x;
    if (j < l) {
        const int yj = p.y[(size_t)r * g + j];
        bool accept;
        float pt;
        if (kGreedy) {
            accept = (yj == row_amax[j]);
            pt = accept ? 1.0f : 0.0f;
        } else {
            pt = exp2f(p.target[(size_t)(first + j) * p.V + yj] * c2 - row_lse[j]);
            const float ratio = pt / p.q_tok[(size_t)r * g + j];
            const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)j, (uint32_t)r, ctr_word3(p.cycle, kAccept)),
                                          (uint32_t)(p.seeds[r] & 0xFFFFFFFFu), (uint32_t)(p.seeds[r] >> 32));
            accept = uniform_from_bits(w.x) < ratio;
        }
        s_pt[j] = pt;
        s_acc[j] = accept;
    }
    __syncthreads();
    int n = l;  // accepted drafts: up to the first rejection
    for (int i = 0; i < l; ++i)
        if (!s_acc[i]) { n = i; break; }
    if (j < l && j <= n && p.p_tok) p.p_tok[(size_t)r * g + j] = s_pt[j];
    int32_t* out = p.out_tokens + (size_t)r * (g + 1);
    if (j <= g && j != n) out[j] = j < n ? p.y[(size_t)r * g + j] : -1;
    if (j == 0) {
        p.n_acc[r] = n;
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
    const long long units = (long long)p.max_rows * p.nsub;  // at most: the rows in use are read on the device
    if (units > 0) {
        int dev = 0, n_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaGetLastError();
        // enough resident warps to keep each SM's share of the stream in flight
        const long long warps = std::min<long long>(units, 24LL * n_sm);
        const unsigned grid1 = (unsigned)((warps * 32 + kStatThreads - 1) / kStatThreads);
        if (p.greedy) {
            verify_stats_kernel<true><<<grid1, kStatThreads, 0, stream>>>(p);
            verify_decide_kernel<true><<<p.R, kStatThreads, 0, stream>>>(p);
        } else {
            verify_stats_kernel<false><<<grid1, kStatThreads, 0, stream>>>(p);
            verify_decide_kernel<false><<<p.R, kStatThreads, 0, stream>>>(p);
        }
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

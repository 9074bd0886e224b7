// draft_simt.cu -- Markov-head block draft on the CUDA cores.
//
// "DSpark explainer" (papers.franksyz.com topic 31) sections 6-7 and llama.cpp
// PR 25173 (draft-dspark): per block position k the drafter's logits are
// U_k + W2 . W1[prev], prev = the anchor at k = 0 and the token drafted at
// k - 1 afterwards, sampled left to right.
//
// This path handles every element type and shape (fp32 factors, ranks that
// are not multiples of 64, ...).  Per position k, two launches:
//   draft_bias_simt    bias[r][v] = sum_j W2[v][j] * W1[prev_r][j], fp32, tiles
//                      of 64 vocabulary rows x 16 requests staged in shared memory;
//   draft_sample       one CTA per (request, 8192-entry chunk): logits, the
//                      segments' Gumbel race and picks, running argmax and (max,
//                      sum of exp); the last CTA of a request (counter, no spin)
//                      writes y, q_lse, q_tok.
#include "kernels.cuh"

namespace dspark {
namespace {

constexpr int kBiasTileV = 64;
constexpr int kBiasTileR = 16;
constexpr int kBiasTileK = 64;

// prev token of request r at position k; -1 = no bias; -2 = unusable request.
__device__ __forceinline__ int prev_token(const DraftParams& p, int r, int k) {
    if (k == 0) {
        const int a = p.anchor[r];
        return a >= p.V ? -2 : (a < 0 ? -1 : a);
    }
    const int t = p.y[(size_t)r * p.gamma + k - 1];
    return (t < 0 || t >= p.V) ? -2 : t;
}

__global__ void __launch_bounds__(256) draft_bias_simt_kernel(DraftParams p, int k) {
    __shared__ float Hs[kBiasTileR][kBiasTileK];
    __shared__ float Ws[kBiasTileV][kBiasTileK + 1];
    __shared__ int prev_s[kBiasTileR];
    const int v0 = blockIdx.x * kBiasTileV;
    const int r0 = blockIdx.y * kBiasTileR;
    if (threadIdx.x < kBiasTileR) {
        const int r = r0 + threadIdx.x;
        prev_s[threadIdx.x] = r < p.R ? prev_token(p, r, k) : -1;
    }
    __syncthreads();
    const int tv = threadIdx.x % kBiasTileV;
    const int tr = threadIdx.x / kBiasTileV;  // requests 4*tr .. 4*tr+3 of the tile
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int j0 = 0; j0 < p.rank; j0 += kBiasTileK) {
        for (int e = threadIdx.x; e < kBiasTileR * kBiasTileK; e += blockDim.x) {
            const int i = e / kBiasTileK, j = e % kBiasTileK;
            const int pr = prev_s[i];
            Hs[i][j] = (pr >= 0 && j0 + j < p.rank)
                           ? load_elem(p.W1, p.w_dtype, (size_t)pr * p.rank + j0 + j) : 0.0f;
        }
        for (int e = threadIdx.x; e < kBiasTileV * kBiasTileK; e += blockDim.x) {
            const int i = e / kBiasTileK, j = e % kBiasTileK;
            Ws[i][j] = (v0 + i < p.V && j0 + j < p.rank)
                           ? load_elem(p.W2, p.w_dtype, (size_t)(v0 + i) * p.rank + j0 + j) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int j = 0; j < kBiasTileK; ++j) {
            const float w = Ws[tv][j];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, Hs[4 * tr + i][j], acc[i]);
        }
        __syncthreads();
    }
    const int v = v0 + tv;
    if (v < p.V) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + 4 * tr + i;
            if (r < p.R) p.bias[(size_t)r * p.V + v] = acc[i];
        }
    }
}

__device__ __forceinline__ void draft_block_reduce(float& score, int& idx, float& s_at,
                                                   float& m, float& sum) {
    __shared__ float a_sc[32], a_sa[32], a_m[32], a_su[32];
    __shared__ int a_ix[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float sc = shfl_xor(score, o), sa = shfl_xor(s_at, o);
        const float m2 = shfl_xor(m, o), su = shfl_xor(sum, o);
        const int ix = shfl_xor(idx, o);
        if (better(sc, ix, score, idx)) { score = sc; idx = ix; s_at = sa; }
        lse_merge(m, sum, m2, su);
    }
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { a_sc[w] = score; a_ix[w] = idx; a_sa[w] = s_at; a_m[w] = m; a_su[w] = sum; }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        score = lane < nw ? a_sc[lane] : -INFINITY;
        idx = lane < nw ? a_ix[lane] : INT_MAX;
        s_at = lane < nw ? a_sa[lane] : 0.0f;
        m = lane < nw ? a_m[lane] : -INFINITY;
        sum = lane < nw ? a_su[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float sc = shfl_xor(score, o), sa = shfl_xor(s_at, o);
            const float m2 = shfl_xor(m, o), su = shfl_xor(sum, o);
            const int ix = shfl_xor(idx, o);
            if (better(sc, ix, score, idx)) { score = sc; idx = ix; s_at = sa; }
            lse_merge(m, sum, m2, su);
        }
    }
}

template <bool kGreedy>
__global__ void __launch_bounds__(kDraftThreads) draft_sample_kernel(DraftParams p, int k) {
    __shared__ int s_last;
    const int r = blockIdx.x / p.nchunk;
    const int chunk = blockIdx.x - r * p.nchunk;
    const int g = p.gamma;
    const size_t rk = (size_t)r * g + k;
    if (prev_token(p, r, k) == -2) {  // bad anchor: the whole request is unusable
        if (chunk == 0 && threadIdx.x == 0) {
            p.y[rk] = -1;
            if (p.q_lse) p.q_lse[rk] = NAN;
            if (p.q_tok) p.q_tok[rk] = NAN;
            report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
        }
        return;
    }
    const int V = p.V;
    const int v0 = chunk * kDraftChunk;
    const int v1 = min(V, v0 + kDraftChunk);
    const float* brow = p.bias + (size_t)r * V;
    float* qrow = p.q_logits ? p.q_logits + rk * V : nullptr;
    PhiloxKey K;
    if (!kGreedy) K = philox_key(p.seeds[r]);
    const uint32_t w3 = ctr_word3(p.cycle, kDraftGumbel);

    float score = -INFINITY, s_at = 0.0f, m = -INFINITY, sum = 0.0f;
    int idx = INT_MAX;
    if (kGreedy) {
        for (int v = v0 + threadIdx.x; v < v1; v += kDraftThreads) {
            const float s = load_elem(p.U, p.u_dtype, rk * V + v) + brow[v];
            if (qrow) qrow[v] = s;
            if (better(s, v, score, idx)) { score = s; idx = v; s_at = s; }
        }
    } else {
        // Gumbel-max with its noise built per 16-entry segment: the segment's race
        // value log W - log(-log u) and, for its pick, the first entry whose running
        // weight passes a W (u, a: words 2 h, 2 h + 1 of the counter 4 (s / 8) + s % 4,
        // h = (s / 4) % 2).  Each segment offers its pick with its race value; the
        // best offer over the vocabulary is the draw.
        for (int sg = (v0 >> 4) + (int)threadIdx.x; 16 * sg < v1; sg += kDraftThreads) {
            const uint4 wd = philox4x32_10(
                make_uint4((uint32_t)(4 * (sg >> 3) + (sg & 3)), (uint32_t)k, (uint32_t)r, w3), K);
            const bool hi = (sg >> 2) & 1;
            const float u = uniform_from_bits(hi ? wd.z : wd.x);
            const float a = uniform_from_bits(hi ? wd.w : wd.y);
            float sv[16];
            float ms = -INFINITY;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int v = 16 * sg + c;
                float s = -INFINITY;
                if (v < v1) {
                    s = (load_elem(p.U, p.u_dtype, rk * V + v) + brow[v]) * p.invT;
                    if (qrow) qrow[v] = s;
                }
                sv[c] = s;
                ms = fmaxf(ms, s);
            }
            if (!(ms > -INFINITY)) continue;  // nothing finite in the segment
            float w = 0.0f;
#pragma unroll
            for (int c = 0; c < 16; ++c) w += expf(sv[c] - ms);
            lse_merge(m, sum, ms, w);
            const float race = ms + logf(w) + gumbel_from_uniform(u);
            const float target = a * w;
            float run = 0.0f;
            int pick = -1, last = 0;
            float s_pick = sv[0];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float wc = expf(sv[c] - ms);
                run += wc;
                if (wc > 0.0f && pick < 0) last = c;
                if (pick < 0 && run > target) { pick = c; s_pick = sv[c]; }
            }
            if (pick < 0) {
                pick = last;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c == last) s_pick = sv[c];
            }
            if (better(race, 16 * sg + pick, score, idx)) { score = race; idx = 16 * sg + pick; s_at = s_pick; }
        }
    }
    draft_block_reduce(score, idx, s_at, m, sum);
    if (threadIdx.x == 0) {
        DraftPartial dp;
        dp.score = score; dp.idx = idx; dp.s_at = s_at; dp.m = m; dp.sum = sum;
        dp.pad[0] = dp.pad[1] = dp.pad[2] = 0.0f;
        p.parts[(size_t)r * p.nchunk + chunk] = dp;
        __threadfence();
        s_last = (atomicAdd(p.cnt + r, 1) == p.nchunk - 1);
    }
    __syncthreads();
    if (!s_last || threadIdx.x != 0) return;
    __threadfence();
    float fs = -INFINITY, fa = 0.0f, fm = -INFINITY, fsum = 0.0f;
    int fi = INT_MAX;
    for (int c = 0; c < p.nchunk; ++c) {
        const DraftPartial* q = p.parts + (size_t)r * p.nchunk + c;
        const float sc = __ldcg(&q->score), sa = __ldcg(&q->s_at);
        const int ix = __ldcg(&q->idx);
        if (better(sc, ix, fs, fi)) { fs = sc; fi = ix; fa = sa; }
        lse_merge(fm, fsum, __ldcg(&q->m), __ldcg(&q->sum));
    }
    if (fi >= p.V) {  // no finite score at all (NaN logits): unusable request
        p.y[rk] = -1;
        if (p.q_lse) p.q_lse[rk] = NAN;
        if (p.q_tok) p.q_tok[rk] = NAN;
        report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
        p.cnt[r] = 0;
        return;
    }
    p.y[rk] = fi;
    if (!kGreedy) {
        const float lse = fm + logf(fsum);
        if (p.q_lse) p.q_lse[rk] = lse;
        if (p.q_tok) p.q_tok[rk] = expf(fa - lse);
    }
    p.cnt[r] = 0;  // ready for the next position
}

__global__ void clear_counters_kernel(int* cnt, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) cnt[i] = 0;
}

}  // namespace

cudaError_t launch_draft_simt(const DraftParams& p, cudaStream_t stream) {
    clear_counters_kernel<<<(p.R + 255) / 256, 256, 0, stream>>>(p.cnt, p.R);
    const dim3 bias_grid((p.V + kBiasTileV - 1) / kBiasTileV, (p.R + kBiasTileR - 1) / kBiasTileR);
    const unsigned sample_grid = (unsigned)((long long)p.R * p.nchunk);
    for (int k = 0; k < p.gamma; ++k) {
        draft_bias_simt_kernel<<<bias_grid, 256, 0, stream>>>(p, k);
        if (p.greedy) draft_sample_kernel<true><<<sample_grid, kDraftThreads, 0, stream>>>(p, k);
        else draft_sample_kernel<false><<<sample_grid, kDraftThreads, 0, stream>>>(p, k);
    }
    return cudaGetLastError();
}

}  // namespace dspark

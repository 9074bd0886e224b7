// select.cu -- survival, capacity planning and prefix-closed top-K selection,
// and the commit lengths.
//
// "DSpark explainer" (papers.franksyz.com topic 31): section 5 (the value of a
// suffix position is the product of the conditional acceptance rates), section
// 8 (survival a[r,k] from the confidences c[r,k]), section 9 (prefix-closed
// selection maximising predicted output x SPS(B); the theoretical greedy stops
// when Theta stops improving), section 10 (the physical capacity comes from the
// confidences of an earlier step, the top-K of the current a fills it),
// sections 2 and 11 (commit the accepted prefix plus one token, roll back the
// rest).
//
// The selection runs in one CTA of 1024 threads: R * gamma <= 8192 candidates.
//   1. a = running fp32 product of c along k (one thread per request);
//   2. a stable LSD radix sort of the candidates by the bits of a (31 one-bit
//      split passes, largest first); candidates enter in (k, r) order, so equal
//      a keep position-then-request order and every top-n set is prefix-closed;
//   3. an inclusive fp64 scan of the sorted a gives sum-of-best-n for every n;
//   4. the capacity rule picks n; positions < n of the sorted list are chosen.
#include "kernels.cuh"

namespace dspark {
namespace {

constexpr int kNT = kSelectThreads;

// Exclusive scan of one int per thread over the CTA; returns the total in *tot.
__device__ __forceinline__ int block_exclusive_scan(int x, int* tot, int* warp_sums) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_sums[lane] = wi - ws;  // exclusive
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const int res = warp_sums[w] + incl - x;
    *tot = warp_sums[32];
    __syncthreads();
    return res;
}

__device__ __forceinline__ double block_exclusive_scan_d(double x, double* tot, double* warp_sums) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    double incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        const double ws = warp_sums[lane];
        double wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_sums[lane] = wi - ws;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const double res = warp_sums[w] + incl - x;
    *tot = warp_sums[32];
    __syncthreads();
    return res;
}

struct SelectSmem {
    uint32_t key[2][kSelectMaxItems];  // float bits of a (non-negative: order-preserving)
    uint16_t id[2][kSelectMaxItems];   // candidate id = k * R + r
    double prefix[kSelectMaxItems + 1];  // prefix[n] = sum of the n best a
    int l[kSelectMaxItems];
    int cs[kSelectMaxSteps];
    float sp[kSelectMaxSteps];
    int warp_i[33];
    double warp_d[33];
    int flag;
    int n_sel;
};

// Fill keys from confidences (computing the survival products), sort, scan.
// Returns false if a confidence is outside [0, 1].  Leaves the sorted ids in
// buffer 0 and prefix sums in sm.prefix.  Without do_sort (the selection takes
// every candidate or none, so order does not matter) it stops after the
// products.
__device__ bool survival_sort_scan(SelectSmem& sm, const float* c, float* a_out, int R, int gamma,
                                   bool do_sort = true) {
    const int N = R * gamma;
    if (threadIdx.x == 0) sm.flag = 0;
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += kNT) {
        // the request's confidences, all loads in flight at once (gamma <= 16)
        float cv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) cv[k] = k < gamma ? c[(size_t)r * gamma + k] : 1.0f;
        float run = 1.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k >= gamma) break;
            const float ck = cv[k];
            if (!(ck >= 0.0f && ck <= 1.0f)) atomicOr(&sm.flag, 1);
            run = (k == 0) ? ck : run * ck;
            const int idn = k * R + r;
            sm.key[0][idn] = __float_as_uint(run);
            sm.id[0][idn] = (uint16_t)idn;
            if (a_out) a_out[(size_t)r * gamma + k] = run;
        }
    }
    __syncthreads();
    if (sm.flag) return false;
    if (!do_sort) return true;

    // stable split passes, one per bit, ones (larger) first; blocked layout over
    // all threads (thread t holds candidates t * ipt .. + ipt - 1, in order)
    int src = 0;
    const int ipt = (N + kNT - 1) / kNT;
    const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
    for (int bit = 0; bit < 31; ++bit) {
        int ones = 0;
        for (int i = lo; i < hi; ++i) ones += (sm.key[src][i] >> bit) & 1u;
        int total1;
        const int ones_before = block_exclusive_scan(ones, &total1, sm.warp_i);
        int o = ones_before;
        int z = total1 + (lo - ones_before);
        for (int i = lo; i < hi; ++i) {
            const uint32_t kk = sm.key[src][i];
            const int dst = ((kk >> bit) & 1u) ? o++ : z++;
            sm.key[src ^ 1][dst] = kk;
            sm.id[src ^ 1][dst] = sm.id[src][i];
        }
        __syncthreads();
        src ^= 1;
    }
    // 31 passes: the result sits in buffer 1; move it to buffer 0
    for (int i = threadIdx.x; i < N; i += kNT) {
        sm.key[0][i] = sm.key[1][i];
        sm.id[0][i] = sm.id[1][i];
    }
    __syncthreads();
    // inclusive prefix sums of the sorted a in fp64, blocked per thread
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += (double)__uint_as_float(sm.key[0][i]);
    double tot;
    double run = block_exclusive_scan_d(local, &tot, sm.warp_d);
    if (threadIdx.x == 0) sm.prefix[0] = 0.0;
    for (int i = lo; i < hi; ++i) {
        run += (double)__uint_as_float(sm.key[0][i]);
        sm.prefix[i + 1] = run;
    }
    __syncthreads();
    return true;
}

__global__ void __launch_bounds__(kNT) select_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
    const int R = p.R, gamma = p.gamma, N = R * gamma;

    // capture sizes sorted ascending (with their step rates)
    if (threadIdx.x == 0 && p.mode != DSPARK_SELECT_FIXED) {
        for (int i = 0; i < p.n_steps; ++i) { sm.cs[i] = p.capture_sizes[i]; sm.sp[i] = p.sps[i]; }
        for (int i = 1; i < p.n_steps; ++i)
            for (int j = i; j > 0 && sm.cs[j - 1] > sm.cs[j]; --j) {
                const int t = sm.cs[j]; sm.cs[j] = sm.cs[j - 1]; sm.cs[j - 1] = t;
                const float f = sm.sp[j]; sm.sp[j] = sm.sp[j - 1]; sm.sp[j - 1] = f;
            }
    }
    __syncthreads();

    bool good = true;
    int n = 0;
    if (p.mode == DSPARK_SELECT_HISTORY) {
        good = survival_sort_scan(sm, p.c_hist, nullptr, R, gamma);
    } else {
        const int n_fixed = min(p.K_cap - R, N);
        const bool all_or_none = p.mode == DSPARK_SELECT_FIXED && (n_fixed == 0 || n_fixed == N);
        good = survival_sort_scan(sm, p.c, p.a, R, gamma, !all_or_none);
    }
    if (good && (p.mode == DSPARK_SELECT_HISTORY || p.mode == DSPARK_SELECT_CURRENT)) {
        if (threadIdx.x == 0) {
            double best = -1.0;
            int best_S = -1, best_n = 0;
            for (int i = 0; i < p.n_steps; ++i) {
                const int S = sm.cs[i];
                if (S < R) continue;
                const int ni = min(min(S, p.K_cap) - R, N);
                const double th = (double)sm.sp[i] * ((double)R + sm.prefix[ni]);
                if (best_S < 0 || th > best) { best = th; best_S = S; best_n = ni; }
            }
            sm.n_sel = best_S < 0 ? 0 : best_n;
        }
        __syncthreads();
        n = sm.n_sel;
        if (p.mode == DSPARK_SELECT_HISTORY) good = survival_sort_scan(sm, p.c, p.a, R, gamma, n != 0 && n != N);
    } else if (good && p.mode == DSPARK_SELECT_FIRST_STOP) {
        // Theta(n) for every n in parallel; the answer is the first n whose
        // successor is not strictly better (or infeasible).
        if (threadIdx.x == 0) sm.n_sel = INT_MAX;
        __syncthreads();
        auto pad = [&](int B) {  // index of the smallest capture size >= B, or -1
            int lo = 0, hi = p.n_steps;
            while (lo < hi) { const int mid = (lo + hi) >> 1; if (sm.cs[mid] >= B) hi = mid; else lo = mid + 1; }
            return lo < p.n_steps ? lo : -1;
        };
        const int p0 = pad(R);
        if (p0 < 0) {
            if (threadIdx.x == 0) sm.n_sel = 0;
        } else {
            for (int m = threadIdx.x; m < N; m += kNT) {
                // may we go from m to m + 1 candidates?
                const int B0 = R + m, B1 = R + m + 1;
                const int i0 = pad(B0), i1 = pad(B1);
                bool stop = (B1 > p.K_cap) || i1 < 0;
                if (!stop) {
                    const double th0 = (double)sm.sp[i0] * ((double)R + sm.prefix[m]);
                    const double th1 = (double)sm.sp[i1] * ((double)R + sm.prefix[m + 1]);
                    stop = !(th1 > th0);
                }
                if (stop) atomicMin(&sm.n_sel, m);
            }
        }
        __syncthreads();
        n = min(sm.n_sel, N);
    } else if (good) {
        n = min(p.K_cap - R, N);
    }
    __syncthreads();
    if (!good) {
        for (int r = threadIdx.x; r < R; r += kNT) p.l[r] = -1;
        for (int r = threadIdx.x; r <= R; r += kNT) p.cu[r] = -1;
        if (threadIdx.x == 0) { p.K_used[0] = -1; report(p.dev_status, DSPARK_ERR_DEVICE_INPUT); }
        return;
    }
    for (int r = threadIdx.x; r < R; r += kNT) sm.l[r] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kNT) atomicAdd(&sm.l[sm.id[0][i] % R], 1);
    __syncthreads();
    // cu_seqlens: exclusive scan of l + 1 (blocked by thread)
    const int per = (R + kNT - 1) / kNT;
    const int lo = min(R, threadIdx.x * per), hi = min(R, lo + per);
    int local = 0;
    for (int r = lo; r < hi; ++r) local += sm.l[r] + 1;
    int tot;
    int run = block_exclusive_scan(local, &tot, sm.warp_i);
    for (int r = lo; r < hi; ++r) {
        p.l[r] = sm.l[r];
        p.cu[r] = run;
        run += sm.l[r] + 1;
    }
    if (threadIdx.x == 0) { p.cu[R] = tot; p.K_used[0] = R + n; }
}

__global__ void __launch_bounds__(1024) commit_kernel(const int32_t* n_acc, const int32_t* l, int R,
                                                     int gamma, int32_t* commit_len, int32_t* cu_commit,
                                                     int32_t* discard, int32_t* total, int32_t* dev_status) {
    __shared__ int warp_i[33];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < R; base += blockDim.x) {
        const int r = base + threadIdx.x;
        int cl = 0;
        if (r < R) {
            const int lr = l ? l[r] : gamma;
            const int na = n_acc[r];
            if (na < 0 || na > lr || lr > gamma) {
                report(dev_status, DSPARK_ERR_DEVICE_INPUT);
                commit_len[r] = 0;
                discard[r] = 0;
            } else {
                cl = na + 1;
                commit_len[r] = cl;
                discard[r] = lr - na;
            }
        }
        int tot;
        const int ex = block_exclusive_scan(cl, &tot, warp_i);
        if (r < R) cu_commit[r] = carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        cu_commit[R] = carry;
        if (total) total[0] = carry;
    }
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
    const size_t smem = sizeof(SelectSmem);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<1, kNT, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_commit(const int32_t* n_acc, const int32_t* l, int R, int gamma,
                          int32_t* commit_len, int32_t* cu_commit, int32_t* discard,
                          int32_t* total, int32_t* dev_status, cudaStream_t stream) {
    commit_kernel<<<1, 1024, 0, stream>>>(n_acc, l, R, gamma, commit_len, cu_commit, discard,
                                          total, dev_status);
    return cudaGetLastError();
}

}  // namespace dspark

// calibrate.cu -- sequential temperature scaling of the confidence head.
//
// "DSpark explainer" (papers.franksyz.com topic 31) section 8: the scheduler
// multiplies per-position confidences into survival probabilities, so the
// confidences must be calibrated, which the paper does left to right with a
// post-hoc temperature per position; llama.cpp PR 25173 "Future work" names it
// Sequential Temperature Scaling.  Position k is fitted on the samples that
// reached it (every earlier draft accepted): c_k = sigmoid(z_k / tau_k) is then
// the conditional acceptance rate the survival product multiplies.
//
// With beta = 1 / tau the negative log-likelihood
//   NLL(beta) = sum_i softplus(beta z_i) - y_i beta z_i
// is convex in beta; Newton steps g / h with
//   g = sum_i (sigmoid(beta z_i) - y_i) z_i,  h = sum_i s_i (1 - s_i) z_i^2
// from beta = 1, halving beta whenever a step would leave (0, inf), until the
// step is below 1e-12 of beta (at most 60 steps); beta is then clamped to
// [1e-3, 1e3].  A position that no sample reached keeps tau = 1.
//
// One cooperative launch: up to kCalMaxCtas CTAs per position; every Newton step, each
// CTA sums (g, h) over its share of the samples in fp64, publishes the pair,
// and after a barrier of the position's CTAs every CTA combines the pairs in
// CTA order and takes the same step (so all agree without a second barrier).
// The data (z column and the labels up to k) stay in L2 across the steps.
#include <algorithm>

#include "kernels.cuh"

namespace dspark {
namespace {

constexpr int kCalThreads = 512;
constexpr int kCalMaxIters = 60;

struct CalParams {
    const float* z;            // [N, gamma]
    const uint8_t* accepted;   // [N, gamma]
    int N, gamma, ctas;        // ctas per position
    float* tau;                // [gamma]
    double* nll;               // [gamma] or NULL
    int32_t* count;            // [gamma] or NULL
    int32_t* dev_status;
    double* part;              // [2][gamma][ctas][4] (g, h, nll, count) by step parity
    unsigned* bar;             // [gamma] arrivals per position, zeroed before the launch
    int* abort_word;           // [1], zeroed before the launch
    unsigned long long wait_ns;
};

__device__ __forceinline__ double sigmoid_d(double x) {
    return x >= 0.0 ? 1.0 / (1.0 + exp(-x)) : exp(x) / (1.0 + exp(x));
}
__device__ __forceinline__ double softplus_d(double x) {
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

// Sum of four doubles over the CTA; every thread gets the totals.
__device__ __forceinline__ void block_sum4(double (&v)[4]) {
    __shared__ double sh[kCalThreads / 32][4];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[q] += __shfl_xor_sync(0xFFFFFFFFu, v[q], o);
    if (lane == 0)
#pragma unroll
        for (int q = 0; q < 4; ++q) sh[w][q] = v[q];
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        double t = 0.0;
        for (int i = 0; i < kCalThreads / 32; ++i) t += sh[i][q];
        v[q] = t;
    }
    __syncthreads();
}

// The position's CTAs meet after publishing step `step`'s partial sums
// (arrivals counted on a per-position counter that only grows).  Bounded.
__device__ __forceinline__ bool position_barrier(const CalParams& p, int k, int step) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(p.bar + k, 1u);
        const unsigned target = (unsigned)(p.ctas * (step + 1));
        const uint64_t t0 = global_ns();
        int good = 1;
        for (unsigned it = 1; *reinterpret_cast<volatile unsigned*>(p.bar + k) < target; ++it) {
            if ((it & 31) == 0) {
                if (*reinterpret_cast<volatile int*>(p.abort_word)) { good = 0; break; }
                if (global_ns() - t0 > p.wait_ns) { atomicExch(p.abort_word, 1); good = 0; break; }
            }
        }
        __threadfence();
        ok = good;
    }
    __syncthreads();
    return ok != 0;
}

__global__ void __launch_bounds__(kCalThreads) calibrate_kernel(CalParams p) {
    const int k = blockIdx.x / p.ctas, c = blockIdx.x - k * p.ctas;
    const int g = p.gamma;
    // this CTA's samples: a contiguous share
    const int per = (p.N + p.ctas - 1) / p.ctas;
    const int i0 = min(p.N, c * per), i1 = min(p.N, i0 + per);
    double beta = 1.0;
    int step = 0;
    bool good = true;
    // partial sums over the samples that reached position k at the current beta
    auto sums = [&](bool with_nll, double (&v)[4]) {
        v[0] = v[1] = v[2] = v[3] = 0.0;
        for (int i = i0 + (int)threadIdx.x; i < i1; i += kCalThreads) {
            const uint8_t* a = p.accepted + (size_t)i * g;
            bool reached = true;
            for (int j = 0; j < k; ++j) reached = reached && a[j] != 0;
            if (!reached) continue;
            const double zi = (double)__ldg(p.z + (size_t)i * g + k);
            const double yi = a[k] ? 1.0 : 0.0;
            const double x = beta * zi;
            if (with_nll) {
                v[2] += softplus_d(x) - yi * x;
            } else {
                const double si = sigmoid_d(x);
                v[0] += (si - yi) * zi;
                v[1] += si * (1.0 - si) * zi * zi;
            }
            v[3] += 1.0;
        }
        block_sum4(v);
    };
    auto publish_and_combine = [&](const double (&v)[4], double (&tot)[4]) -> bool {
        double* mine = p.part + (((size_t)(step & 1) * g + k) * p.ctas + c) * 4;
        if (threadIdx.x == 0)
            for (int q = 0; q < 4; ++q) mine[q] = v[q];
        if (!position_barrier(p, k, step)) return false;
        tot[0] = tot[1] = tot[2] = tot[3] = 0.0;
        const double* all = p.part + ((size_t)(step & 1) * g + k) * p.ctas * 4;
        for (int cc = 0; cc < p.ctas; ++cc)
            for (int q = 0; q < 4; ++q) tot[q] += __ldcg(all + cc * 4 + q);
        ++step;
        return true;
    };
    double tot[4] = {0.0, 0.0, 0.0, 0.0};
    for (int it = 0; it < kCalMaxIters; ++it) {
        double v[4];
        sums(false, v);
        if (!(good = publish_and_combine(v, tot))) break;
        if (!(tot[1] > 0.0)) break;  // nothing reached the position (or no curvature)
        const double d = tot[0] / tot[1];
        const double next = beta - d;
        const bool done = fabs(d) <= 1e-12 * beta;
        beta = (next > 0.0 && isfinite(next)) ? next : 0.5 * beta;
        if (done) break;
    }
    const double n_reached = tot[3];
    beta = fmin(1e3, fmax(1e-3, beta));
    double v[4];
    if (good) {
        sums(true, v);
        good = publish_and_combine(v, tot);
    }
    if (c == 0 && threadIdx.x == 0) {
        if (!good) {
            report(p.dev_status, DSPARK_ERR_TIMEOUT);
            return;
        }
        const bool any = n_reached > 0.0;
        p.tau[k] = any ? (float)(1.0 / beta) : 1.0f;
        if (p.nll) p.nll[k] = any ? tot[2] / n_reached : 0.0;
        if (p.count) p.count[k] = (int32_t)n_reached;
    }
}

}  // namespace

size_t calibrate_workspace(int gamma) {
    // partial sums (two step parities) + barrier counters + abort word
    return (size_t)2 * gamma * kCalMaxCtas * 4 * sizeof(double) + 256 + 256;
}

cudaError_t launch_calibrate(const float* z, const uint8_t* accepted, int N, int gamma, float* tau, double* nll,
                             int32_t* count, int32_t* dev_status, void* ws, cudaStream_t stream) {
    int dev = 0, n_sm = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, calibrate_kernel, kCalThreads, 0)) !=
        cudaSuccess)
        return e;
    // every CTA of a position must be resident with the others (they meet at
    // barriers): at most the resident capacity over all positions
    const int cap = n_sm * per_sm;
    int ctas = std::max(1, std::min(kCalMaxCtas, cap / gamma));
    const int want = (N + 4 * kCalThreads - 1) / (4 * kCalThreads);  // at least 4 samples a thread
    ctas = std::max(1, std::min(ctas, want));
    CalParams p;
    p.z = z; p.accepted = accepted; p.N = N; p.gamma = gamma; p.ctas = ctas;
    p.tau = tau; p.nll = nll; p.count = count; p.dev_status = dev_status;
    unsigned char* w = static_cast<unsigned char*>(ws);
    p.part = reinterpret_cast<double*>(w);
    const size_t part_bytes = (size_t)2 * gamma * kCalMaxCtas * 4 * sizeof(double);
    p.bar = reinterpret_cast<unsigned*>(w + part_bytes);
    p.abort_word = reinterpret_cast<int*>(w + part_bytes + 256);
    p.wait_ns = grid_wait_limit_ns();
    if ((e = cudaMemsetAsync(w + part_bytes, 0, 512, stream)) != cudaSuccess) return e;
    void* args[] = {&p};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(calibrate_kernel), dim3(gamma * ctas),
                                    dim3(kCalThreads), args, 0, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dspark

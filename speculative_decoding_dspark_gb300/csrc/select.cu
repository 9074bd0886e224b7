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
// The static cutoffs (modes CONF_CUTOFF and SURVIVAL_CUTOFF) mark each
// request's leading positions that pass the cutoff in the key's top bit, so
// one more split pass sorts the eligible candidates first, in the same order.
// dspark_plan_cycles runs the same selection for many cycles at once, one CTA
// per cycle, with the capacity of cycle t planned on the confidences of cycle
// t - lag, and scores each cycle against the drafts the target would accept.
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

constexpr int kTracks = 16;  // top-n sizes one radix selection finds at once

// Shared memory of one selection: fixed fields, then the per-candidate arrays,
// sized for the call's N = R * gamma candidates (select_smem_bytes) and carved
// by select_carve.
struct SelectSmem {
    uint32_t* key[2];  // [N] float bits of a (non-negative: order-preserving); top bit: eligible
    uint16_t* id[2];   // [N] candidate id = k * R + r
    double* prefix;    // [N + 1] sort path: prefix[n] = sum of the n best a
    uint8_t* sel;      // [N] selection path: candidate chosen (shares prefix's space)
    int* l;            // [R]
    int bins[kTracks][256];
    uint32_t tau[kTracks];   // per track: key of the n-th best candidate
    int need[kTracks];       // per track: the wanted count, then how many keys equal to tau are taken
    int track_n[kTracks];
    double track_sum[kTracks];
    int n_tracks;
    int cs[kSelectMaxSteps];
    float sp[kSelectMaxSteps];
    int warp_i[33];
    double warp_d[33];
    int flag;
    int n_sel;
    int n_elig;
};

__host__ __device__ constexpr size_t sel_align(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline size_t select_smem_bytes(int R, int N) {
    return sel_align(sizeof(SelectSmem)) + 2 * sel_align(sizeof(uint32_t) * (size_t)N) +
           2 * sel_align(sizeof(uint16_t) * (size_t)N) + sel_align(sizeof(double) * ((size_t)N + 1)) +
           sel_align(sizeof(int) * (size_t)R);
}

// Thread 0 points the arrays into the dynamic shared memory after the fixed fields.
__device__ SelectSmem& select_carve(unsigned char* base, int R, int N) {
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(base);
    if (threadIdx.x == 0) {
        unsigned char* q = base + sel_align(sizeof(SelectSmem));
        for (int b = 0; b < 2; ++b) { sm.key[b] = reinterpret_cast<uint32_t*>(q); q += sel_align(sizeof(uint32_t) * (size_t)N); }
        for (int b = 0; b < 2; ++b) { sm.id[b] = reinterpret_cast<uint16_t*>(q); q += sel_align(sizeof(uint16_t) * (size_t)N); }
        sm.prefix = reinterpret_cast<double*>(q);
        sm.sel = q;
        q += sel_align(sizeof(double) * ((size_t)N + 1));
        sm.l = reinterpret_cast<int*>(q);
    }
    __syncthreads();
    return sm;
}

constexpr uint32_t kEligible = 0x80000000u;

__device__ __forceinline__ bool cutoff_mode(int mode) {
    return mode == DSPARK_SELECT_CONF_CUTOFF || mode == DSPARK_SELECT_SURVIVAL_CUTOFF;
}

// Fill keys from confidences (computing the survival products), sort, scan.
// Returns false if a confidence is outside [0, 1].  Leaves the sorted ids in
// buffer 0 and prefix sums in sm.prefix.  Without do_sort (the selection takes
// every candidate or none, so order does not matter) it stops after the
// products.  cutoff (a CONF_CUTOFF or SURVIVAL_CUTOFF mode, else 0) marks the
// eligible candidates, counted in sm.n_elig, and sorts them first.
__device__ bool survival_sort_scan(SelectSmem& sm, const float* c, float* a_out, int R, int gamma,
                                   bool do_sort = true, int cutoff = 0, float conf_min = 0.0f) {
    const int N = R * gamma;
    if (threadIdx.x == 0) { sm.flag = 0; sm.n_elig = 0; }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += kNT) {
        // the request's confidences, all loads in flight at once (gamma <= 16)
        float cv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) cv[k] = k < gamma ? c[(size_t)r * gamma + k] : 1.0f;
        float run = 1.0f;
        bool elig = cutoff != 0;
        int n_e = 0;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k >= gamma) break;
            const float ck = cv[k];
            if (!(ck >= 0.0f && ck <= 1.0f)) atomicOr(&sm.flag, 1);
            run = (k == 0) ? ck : run * ck;
            // a request stays eligible up to its first position failing the cutoff
            elig = elig && ((cutoff == DSPARK_SELECT_CONF_CUTOFF ? ck : run) >= conf_min);
            n_e += elig ? 1 : 0;
            const int idn = k * R + r;
            // -0 keys as +0 (a confidence of -0 is a survival of 0: it ties with +0)
            sm.key[0][idn] = (__float_as_uint(run) & ~kEligible) | (elig ? kEligible : 0u);
            sm.id[0][idn] = (uint16_t)idn;
            if (a_out) a_out[(size_t)r * gamma + k] = run;
        }
        if (n_e) atomicAdd(&sm.n_elig, n_e);
    }
    __syncthreads();
    if (sm.flag) return false;
    if (!do_sort) return true;

    // stable split passes, one per bit, ones (larger) first; blocked layout over
    // all threads (thread t holds candidates t * ipt .. + ipt - 1, in order)
    int src = 0;
    const int ipt = (N + kNT - 1) / kNT;
    const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
    const int n_bits = cutoff ? 32 : 31;
    for (int bit = 0; bit < n_bits; ++bit) {
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
    // an odd number of passes leaves the result in buffer 1; move it to buffer 0
    if (src == 1) {
        for (int i = threadIdx.x; i < N; i += kNT) {
            sm.key[0][i] = sm.key[1][i];
            sm.id[0][i] = sm.id[1][i];
        }
        __syncthreads();
    }
    // inclusive prefix sums of the sorted a in fp64, blocked per thread
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += (double)__uint_as_float(sm.key[0][i] & ~kEligible);
    double tot;
    double run = block_exclusive_scan_d(local, &tot, sm.warp_d);
    if (threadIdx.x == 0) sm.prefix[0] = 0.0;
    for (int i = lo; i < hi; ++i) {
        run += (double)__uint_as_float(sm.key[0][i] & ~kEligible);
        sm.prefix[i + 1] = run;
    }
    __syncthreads();
    return true;
}

// Radix selection without a sort: for every track t < sm.n_tracks, the key
// tau[t] of the track_n[t]-th best candidate (1 <= track_n[t] < N) among the
// keys sm.key[0][0 .. N) in candidate order, and need[t] = how many of the
// candidates whose key equals tau[t] the best track_n[t] take (the earliest in
// candidate order, which is position then request: the tie order).  Four
// passes over 8-bit digits, most significant first; each pass counts the
// candidates that agree with a track's digits so far into that track's 256
// bins, and one warp per track walks its bins from the top.
__device__ void radix_select(SelectSmem& sm, int N) {
    const int nt = sm.n_tracks;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < nt) { sm.tau[threadIdx.x] = 0u; sm.need[threadIdx.x] = sm.track_n[threadIdx.x]; }
    const int ipt = (N + kNT - 1) / kNT;
    const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
    for (int d = 0; d < 4; ++d) {
        const int shift = 24 - 8 * d;
        for (int b = threadIdx.x; b < nt * 256; b += kNT) (&sm.bins[0][0])[b] = 0;
        __syncthreads();
        for (int i = lo; i < hi; ++i) {
            const uint32_t key = sm.key[0][i];
            for (int t = 0; t < nt; ++t)
                if (d == 0 || (key >> (shift + 8)) == (sm.tau[t] >> (shift + 8)))
                    atomicAdd(&sm.bins[t][(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp < nt) {
            // lane L holds bins 255 - 8L - j (j = 0..7): the lanes in order walk the bins from the top
            int c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { c[j] = sm.bins[warp][255 - 8 * lane - j]; sum += c[j]; }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const int need = sm.need[warp];
            const int before = incl - sum;
            if (before < need && need <= incl) {  // exactly one lane
                int acc = before, j = 0;
                while (acc + c[j] < need) { acc += c[j]; ++j; }
                sm.tau[warp] |= (uint32_t)(255 - 8 * lane - j) << shift;
                sm.need[warp] = need - acc;
            }
        }
        __syncthreads();
    }
}

// Sum of the track_n[t] best survivals for every track (fixed-order fp64
// reduction, the same on every call): those above tau plus need copies of tau.
__device__ void track_sums(SelectSmem& sm, int N) {
    const int nt = sm.n_tracks;
    const int ipt = (N + kNT - 1) / kNT;
    const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
    for (int t = 0; t < nt; ++t) {
        const uint32_t tau = sm.tau[t];
        double local = 0.0;
        for (int i = lo; i < hi; ++i) {
            const uint32_t key = sm.key[0][i];
            if (key > tau) local += (double)__uint_as_float(key & ~kEligible);
        }
        double tot;
        block_exclusive_scan_d(local, &tot, sm.warp_d);
        if (threadIdx.x == 0)
            sm.track_sum[t] = tot + (double)sm.need[t] * (double)__uint_as_float(tau & ~kEligible);
        __syncthreads();
    }
}

// Mark the n best candidates of the current keys in sm.sel (0 < n < N):
// those above the n-th best key and the earliest ones equal to it.
__device__ void mark_best(SelectSmem& sm, int N, int n) {
    if (threadIdx.x == 0) { sm.n_tracks = 1; sm.track_n[0] = n; }
    __syncthreads();
    radix_select(sm, N);
    const uint32_t tau = sm.tau[0];
    const int take_eq = sm.need[0];
    const int ipt = (N + kNT - 1) / kNT;
    const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
    int eq = 0;
    for (int i = lo; i < hi; ++i) eq += sm.key[0][i] == tau;
    int tot;
    int rank = block_exclusive_scan(eq, &tot, sm.warp_i);
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = sm.key[0][i];
        bool take = key > tau;
        if (key == tau) take = rank++ < take_eq;
        sm.sel[i] = take ? 1 : 0;
    }
    __syncthreads();
}

// Where one selection reads and writes: the current and the planning
// confidences, the mode, and the outputs (a and cu may be NULL).
struct SelectIo {
    const float* c;
    const float* c_hist;
    int mode;
    float* a;
    int32_t* l;
    int32_t* cu;
    int32_t* K_used;
};

// The selection of one cycle by the whole CTA.  Leaves each request's length
// in sm.l and returns the number of selected candidates n, or -1 after
// reporting a bad confidence (the outputs are then -1).
__device__ int select_body(SelectSmem& sm, const SelectParams& p, const SelectIo& io, bool sizes_loaded) {
    const int R = p.R, gamma = p.gamma, N = R * gamma;
    const int mode = io.mode;

    // capture sizes sorted ascending (with their step rates)
    if (!sizes_loaded && threadIdx.x == 0 && mode >= DSPARK_SELECT_HISTORY && mode <= DSPARK_SELECT_FIRST_STOP) {
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
    // capacity from a survival plan (HISTORY: an earlier cycle's; CURRENT: this
    // one's): the sums of the n_S best survivals for the capture sizes by radix
    // selection, no sort (the sort path stays for the first-stop greedy, which
    // needs the sum for every n, and for more distinct sizes than tracks)
    auto plan_sizes = [&]() -> bool {  // false: too many distinct sizes for the tracks
        if (threadIdx.x == 0) {
            int nt = 0;
            bool fits = true;
            for (int i = 0; i < p.n_steps; ++i) {
                const int S = sm.cs[i];
                if (S < R) continue;
                const int ni = min(min(S, p.K_cap) - R, N);
                if (ni <= 0 || ni >= N) continue;
                bool seen = false;
                for (int t = 0; t < nt; ++t) seen = seen || sm.track_n[t] == ni;
                if (seen) continue;
                if (nt == kTracks) { fits = false; break; }
                sm.track_n[nt++] = ni;
            }
            sm.n_tracks = fits ? nt : -1;
        }
        __syncthreads();
        return sm.n_tracks >= 0;
    };
    auto choose_capacity = [&](bool sorted) {
        // sorted: sums from sm.prefix; else from the tracks (and the total for n = N)
        double total = 0.0;
        if (!sorted) {
            const int ipt = (N + kNT - 1) / kNT;
            const int lo = min(N, threadIdx.x * ipt), hi = min(N, lo + ipt);
            double local = 0.0;
            for (int i = lo; i < hi; ++i) local += (double)__uint_as_float(sm.key[0][i] & ~kEligible);
            block_exclusive_scan_d(local, &total, sm.warp_d);
            if (sm.n_tracks > 0) {
                radix_select(sm, N);
                track_sums(sm, N);
            }
        }
        if (threadIdx.x == 0) {
            double best = -1.0;
            int best_S = -1, best_n = 0;
            for (int i = 0; i < p.n_steps; ++i) {
                const int S = sm.cs[i];
                if (S < R) continue;
                const int ni = min(min(S, p.K_cap) - R, N);
                double top = 0.0;
                if (sorted) {
                    top = sm.prefix[ni];
                } else if (ni >= N) {
                    top = total;
                } else if (ni > 0) {
                    for (int t = 0; t < sm.n_tracks; ++t)
                        if (sm.track_n[t] == ni) top = sm.track_sum[t];
                }
                const double th = (double)sm.sp[i] * ((double)R + top);
                if (best_S < 0 || th > best) { best = th; best_S = S; best_n = ni; }
            }
            sm.n_sel = best_S < 0 ? 0 : best_n;
        }
        __syncthreads();
        return sm.n_sel;
    };
    bool sorted = false;  // the selection reads the sorted candidate ids
    if (mode == DSPARK_SELECT_HISTORY || mode == DSPARK_SELECT_CURRENT) {
        const float* plan_c = mode == DSPARK_SELECT_HISTORY ? io.c_hist : io.c;
        const bool fits = plan_sizes();
        good = survival_sort_scan(sm, plan_c, mode == DSPARK_SELECT_CURRENT ? io.a : nullptr, R, gamma, !fits);
        if (good) n = choose_capacity(!fits);
        if (good && mode == DSPARK_SELECT_HISTORY) {
            good = survival_sort_scan(sm, io.c, io.a, R, gamma, false);
        } else if (good && !fits && n != 0 && n != N) {
            sorted = true;  // CURRENT on the sort path: the ids are sorted already
        }
    } else if (mode == DSPARK_SELECT_FIRST_STOP) {
        good = survival_sort_scan(sm, io.c, io.a, R, gamma, true);
        sorted = true;
        if (good) {
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
        }
    } else {
        good = survival_sort_scan(sm, io.c, io.a, R, gamma, false, cutoff_mode(mode) ? mode : 0, p.conf_min);
        if (good) n = cutoff_mode(mode) ? min(sm.n_elig, p.K_cap - R) : min(p.K_cap - R, N);
    }
    __syncthreads();
    if (!good) {
        for (int r = threadIdx.x; r < R; r += kNT) io.l[r] = -1;
        if (io.cu)
            for (int r = threadIdx.x; r <= R; r += kNT) io.cu[r] = -1;
        if (threadIdx.x == 0) { io.K_used[0] = -1; report(p.dev_status, DSPARK_ERR_DEVICE_INPUT); }
        return -1;
    }
    if (sorted) {
        for (int r = threadIdx.x; r < R; r += kNT) sm.l[r] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kNT) atomicAdd(&sm.l[sm.id[0][i] % R], 1);
    } else {
        // the n best current candidates (every one or none without a selection);
        // the set is prefix-closed, so l[r] counts request r's chosen positions
        if (n > 0 && n < N) mark_best(sm, N, n);
        for (int r = threadIdx.x; r < R; r += kNT) {
            int cnt = 0;
            if (n >= N) cnt = gamma;
            else if (n > 0)
                for (int k = 0; k < gamma; ++k) cnt += sm.sel[k * R + r];
            sm.l[r] = cnt;
        }
    }
    __syncthreads();
    // cu_seqlens: exclusive scan of l + 1 (blocked by thread)
    const int per = (R + kNT - 1) / kNT;
    const int lo = min(R, threadIdx.x * per), hi = min(R, lo + per);
    int local = 0;
    for (int r = lo; r < hi; ++r) local += sm.l[r] + 1;
    int tot;
    int run = block_exclusive_scan(local, &tot, sm.warp_i);
    for (int r = lo; r < hi; ++r) {
        io.l[r] = sm.l[r];
        if (io.cu) io.cu[r] = run;
        run += sm.l[r] + 1;
    }
    if (threadIdx.x == 0) {
        if (io.cu) io.cu[R] = tot;
        io.K_used[0] = R + n;
    }
    return n;
}

__global__ void __launch_bounds__(kNT) select_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem& sm = select_carve(smem_raw, p.R, p.R * p.gamma);
    SelectIo io;
    io.c = p.c; io.c_hist = p.c_hist; io.mode = p.mode;
    io.a = p.a; io.l = p.l; io.cu = p.cu; io.K_used = p.K_used;
    select_body(sm, p, io, false);
}

// The fixed capacity when it admits every candidate (K_cap - R >= R * gamma):
// no ranking is needed, every request verifies all gamma drafts.  The same
// outputs as select_body for that case (survival a, l = gamma, cu_seqlens,
// K_used = R + R * gamma, or -1 everywhere after a confidence outside [0, 1]),
// from a kernel small enough that its code is fetched quickly.
__global__ void __launch_bounds__(kNT) select_all_kernel(SelectParams p) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    const int R = p.R, gamma = p.gamma;
    for (int r = threadIdx.x; r < R; r += kNT) {
        float cv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) cv[k] = k < gamma ? p.c[(size_t)r * gamma + k] : 1.0f;
        float run = 1.0f;
        bool ok = true;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k >= gamma) break;
            ok = ok && (cv[k] >= 0.0f && cv[k] <= 1.0f);
            run = (k == 0) ? cv[k] : run * cv[k];
            if (p.a) p.a[(size_t)r * gamma + k] = run;
        }
        if (!ok) bad = 1;
    }
    __syncthreads();
    const bool good = !bad;
    for (int r = threadIdx.x; r <= R; r += kNT) {
        if (r < R) p.l[r] = good ? gamma : -1;
        if (p.cu) p.cu[r] = good ? r * (gamma + 1) : -1;
    }
    if (threadIdx.x == 0) {
        p.K_used[0] = good ? R + R * gamma : -1;
        if (!good) report(p.dev_status, DSPARK_ERR_DEVICE_INPUT);
    }
}

// One cycle of a planning run per CTA (blockIdx.x = cycle t): the selection
// of c_seq[t] (capacity from c_seq[t - lag] in HISTORY mode; K_cap in the
// first lag cycles), then the cycle's predicted and achieved Theta, accepted
// drafts and wasted verify rows.
__global__ void __launch_bounds__(kNT) plan_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem& sm = select_carve(smem_raw, p.R, p.R * p.gamma);
    const int t = blockIdx.x;
    const int R = p.R, gamma = p.gamma;
    const size_t rg = (size_t)R * gamma;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_steps; ++i) { sm.cs[i] = p.capture_sizes[i]; sm.sp[i] = p.sps[i]; }
        for (int i = 1; i < p.n_steps; ++i)
            for (int j = i; j > 0 && sm.cs[j - 1] > sm.cs[j]; --j) {
                const int tt = sm.cs[j]; sm.cs[j] = sm.cs[j - 1]; sm.cs[j - 1] = tt;
                const float f = sm.sp[j]; sm.sp[j] = sm.sp[j - 1]; sm.sp[j - 1] = f;
            }
    }
    __syncthreads();
    SelectIo io;
    io.c = p.c + (size_t)t * rg;
    io.mode = p.mode;
    io.c_hist = nullptr;
    if (p.mode == DSPARK_SELECT_HISTORY) {
        if (t >= p.lag) io.c_hist = p.c + (size_t)(t - p.lag) * rg;
        else io.mode = DSPARK_SELECT_FIXED;
    }
    io.a = nullptr;
    io.l = p.l + (size_t)t * R;
    io.cu = nullptr;
    io.K_used = p.K_used + t;
    const int n = select_body(sm, p, io, true);
    double* out = p.stats + (size_t)t * 4;
    if (n < 0) {
        if (threadIdx.x < 4) out[threadIdx.x] = 0.0;
        return;
    }
    // selected survival and the target's verdicts, per request (a recomputed
    // with the same sequential fp32 products)
    double sel = 0.0;
    int acc = 0, wasted = 0;
    for (int r = threadIdx.x; r < R; r += kNT) {
        const int lr = sm.l[r];
        float run = 1.0f;
        for (int k = 0; k < lr; ++k) {
            const float ck = io.c[(size_t)r * gamma + k];
            run = (k == 0) ? ck : run * ck;
            sel += (double)run;
        }
        if (p.n_full) {
            const int na = min(p.n_full[(size_t)t * R + r], lr);
            acc += na;
            wasted += lr - na;
        }
    }
    double sel_tot;
    block_exclusive_scan_d(sel, &sel_tot, sm.warp_d);
    int acc_tot, wasted_tot;
    block_exclusive_scan(acc, &acc_tot, sm.warp_i);
    block_exclusive_scan(wasted, &wasted_tot, sm.warp_i);
    if (threadIdx.x == 0) {
        const int B = R + n;
        double rate = 0.0;  // the smallest capture size >= B
        for (int i = 0; i < p.n_steps; ++i)
            if (sm.cs[i] >= B) { rate = (double)sm.sp[i]; break; }
        out[0] = rate * ((double)R + sel_tot);
        out[1] = p.n_full ? rate * ((double)R + (double)acc_tot) : 0.0;
        out[2] = p.n_full ? (double)acc_tot : 0.0;
        out[3] = p.n_full ? (double)wasted_tot : 0.0;
    }
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
    if (p.mode == DSPARK_SELECT_FIXED && (long long)p.K_cap - p.R >= (long long)p.R * p.gamma) {
        select_all_kernel<<<1, kNT, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const size_t smem = select_smem_bytes(p.R, p.R * p.gamma);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<1, kNT, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_plan(const SelectParams& p, int n_cycles, cudaStream_t stream) {
    const size_t smem = select_smem_bytes(p.R, p.R * p.gamma);
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    plan_kernel<<<n_cycles, kNT, smem, stream>>>(p);
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

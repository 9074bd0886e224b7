// kv.cu -- the paged KV cache's bookkeeping around one verify.
//
// "DSpark explainer" (papers.franksyz.com topic 31) section 11: the target's
// verify writes its candidate rows into temporary pages (or block-table
// entries); after the first rejection only the accepted prefix is promoted to
// committed state and every other candidate's state is released; section 15:
// leaked or double-freed temporary state is among the failure classes.
//
// State: per request its committed length kv_len (tokens) and a row of the
// block table (page b holds positions [b P, (b + 1) P)); committed pages are
// the leading ceil(kv_len / P) entries, the rest -1.  Free pages form a stack
// free_pages[0 .. free_top).
//
//   reserve  request r needs ceil((kv_len + l + 1) / P) - ceil(kv_len / P) more
//            pages for its l + 1 verify rows; the top T = sum of needs pages of
//            the stack go out in request order (request r takes entries
//            free_top - T + o_r ..., o_r = the needs of the requests before it),
//            all or nothing;
//   commit   kv_len += n_acc + 1; the pages past ceil(kv_len / P) held only
//            rejected rows: they go back on the stack in request order and
//            their entries become -1 (entries holding no page are skipped;
//            all or nothing if the stack could not take them).
// Both run in one CTA (the order of the stack is a scan over the requests).
// Every write into the stack is checked against its capacity (pool_pages).
#include "kernels.cuh"

namespace dspark {
namespace {

constexpr int kKvThreads = 1024;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Exclusive scan of one int per thread over the CTA; *tot receives the sum.
__device__ __forceinline__ int kv_scan(int x, int* tot, int* warp_sums) {
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
        const int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_sums[lane] = wi - ws;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const int res = warp_sums[w] + incl - x;
    *tot = warp_sums[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kKvThreads) kv_reserve_kernel(const int32_t* kv_len, const int32_t* l, int R, int P,
                                                                int32_t* bt, int max_blocks, const int32_t* free_pages,
                                                                int32_t* free_top, int pool_pages, int32_t* reserved,
                                                                int32_t* dev_status) {
    __shared__ int warp_sums[33];
    __shared__ int first_bad;  // (lowest failing request << 1) | kind, kind 0 bad length, 1 past max_blocks
    __shared__ long long total;
    if (threadIdx.x == 0) { first_bad = INT_MAX; total = 0; }
    __syncthreads();
    // needs, checks and their total
    for (int base = 0; base < R; base += kKvThreads) {
        const int r = base + threadIdx.x;
        int need = 0;
        if (r < R) {
            const int len = kv_len[r], lr = l[r];
            if (len < 0 || lr < 0 || len > INT_MAX - lr - P) {
                atomicMin(&first_bad, r << 1);
            } else {
                const int want = ceil_div(len + lr + 1, P);
                if (want > max_blocks) atomicMin(&first_bad, (r << 1) | 1);
                else need = want - ceil_div(len, P);
            }
        }
        int tot;
        kv_scan(need, &tot, warp_sums);
        if (threadIdx.x == 0) total += tot;
        __syncthreads();
    }
    const int top = *free_top;
    if (top < 0 || top > pool_pages) {
        if (threadIdx.x == 0) report(dev_status, DSPARK_ERR_DEVICE_INPUT);
        return;
    }
    if (first_bad != INT_MAX || total > top) {
        if (threadIdx.x == 0)
            report(dev_status, (first_bad != INT_MAX && !(first_bad & 1)) ? DSPARK_ERR_DEVICE_INPUT : DSPARK_ERR_CAPACITY);
        return;
    }
    // hand out the top `total` pages of the stack in request order
    const int base_page = top - (int)total;
    int carry = 0;
    for (int base = 0; base < R; base += kKvThreads) {
        const int r = base + threadIdx.x;
        int need = 0, have = 0;
        if (r < R) {
            have = ceil_div(kv_len[r], P);
            need = ceil_div(kv_len[r] + l[r] + 1, P) - have;
        }
        int tot;
        const int o = carry + kv_scan(need, &tot, warp_sums);
        if (r < R) {
            for (int i = 0; i < need; ++i) {
                const int32_t pg = free_pages[base_page + o + i];
                // (a debug build: a page id outside the pool is reported and not handed out)
                bt[(size_t)r * max_blocks + have + i] = IN_BOUNDS(pg >= 0 && pg < pool_pages, dev_status) ? pg : -1;
            }
            if (reserved) reserved[r] = need;
        }
        carry += tot;
    }
    if (threadIdx.x == 0) *free_top = base_page;
}

__global__ void __launch_bounds__(kKvThreads) kv_commit_kernel(int32_t* kv_len, const int32_t* l, const int32_t* n_acc,
                                                               int R, int P, int32_t* bt, int max_blocks,
                                                               int32_t* free_pages, int32_t* free_top, int pool_pages,
                                                               int32_t* dev_status) {
    __shared__ int warp_sums[33];
    __shared__ long long pushes;
    __shared__ int bad;
    if (threadIdx.x == 0) { pushes = 0; bad = 0; }
    const int top = *free_top;
    __syncthreads();  // every thread has read the stack top before it moves
    // the span of request r: kept pages [0, keep), released [keep, held)
    auto span = [&](int r, int& keep, int& held, int& new_len) {
        const int len = kv_len[r], lr = l[r], na = n_acc[r];
        if (len < 0 || lr < 0 || len > INT_MAX - lr - P) {  // unusable lengths: touch nothing
            bad = 1;
            keep = held = 0;
            new_len = len;
            return;
        }
        held = min(max_blocks, ceil_div(len + lr + 1, P));
        const bool ok = na >= 0 && na <= lr;
        if (!ok) bad = 1;
        new_len = len + (ok ? na + 1 : 0);
        keep = ceil_div(new_len, P);
    };
    // the pages that go back, and whether the stack can take them
    for (int base = 0; base < R; base += kKvThreads) {
        const int r = base + threadIdx.x;
        int n = 0;
        if (r < R) {
            int keep, held, new_len;
            span(r, keep, held, new_len);
            for (int b = keep; b < held; ++b) n += bt[(size_t)r * max_blocks + b] >= 0;
        }
        int tot;
        kv_scan(n, &tot, warp_sums);
        if (threadIdx.x == 0) pushes += tot;
        __syncthreads();
    }
    if (top < 0 || top + pushes > pool_pages) {
        if (threadIdx.x == 0) report(dev_status, DSPARK_ERR_DEVICE_INPUT);
        return;
    }
    if (threadIdx.x == 0 && bad) report(dev_status, DSPARK_ERR_DEVICE_INPUT);
    int carry = 0;
    for (int base = 0; base < R; base += kKvThreads) {
        const int r = base + threadIdx.x;
        int n = 0, keep = 0, held = 0, new_len = 0;
        if (r < R) {
            span(r, keep, held, new_len);
            for (int b = keep; b < held; ++b) n += bt[(size_t)r * max_blocks + b] >= 0;
        }
        int tot;
        int o = top + carry + kv_scan(n, &tot, warp_sums);
        if (r < R) {
            for (int b = keep; b < held; ++b) {
                int32_t* e = bt + (size_t)r * max_blocks + b;
                if (*e >= 0 && IN_BOUNDS(*e < pool_pages, dev_status)) free_pages[o++] = *e;
                *e = -1;
            }
            kv_len[r] = new_len;
        }
        carry += tot;
    }
    if (threadIdx.x == 0) *free_top = top + carry;
}

}  // namespace

cudaError_t launch_kv_reserve(const int32_t* kv_len, const int32_t* l, int R, int P, int32_t* bt, int max_blocks,
                              const int32_t* free_pages, int32_t* free_top, int pool_pages, int32_t* reserved,
                              int32_t* dev_status, cudaStream_t stream) {
    kv_reserve_kernel<<<1, kKvThreads, 0, stream>>>(kv_len, l, R, P, bt, max_blocks, free_pages, free_top, pool_pages,
                                                   reserved, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_kv_commit(int32_t* kv_len, const int32_t* l, const int32_t* n_acc, int R, int P, int32_t* bt,
                             int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages,
                             int32_t* dev_status, cudaStream_t stream) {
    kv_commit_kernel<<<1, kKvThreads, 0, stream>>>(kv_len, l, n_acc, R, P, bt, max_blocks, free_pages, free_top,
                                                  pool_pages, dev_status);
    return cudaGetLastError();
}

}  // namespace dspark

// common.cuh -- device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies on counter
// words 0 and 2, the high halves xor-ed with the other two words and the
// round key, the key advanced by two Weyl increments between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Precomputed round keys of one 64-bit seed (the key schedule does not depend
// on the counter, so a thread drawing many numbers for one request keeps it).
struct PhiloxKey {
    uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
    PhiloxKey K;
    uint32_t a = (uint32_t)(seed & 0xFFFFFFFFu), b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        K.k0[i] = a; K.k1[i] = b;
        a += 0x9E3779B9u; b += 0xBB67AE85u;
    }
    return K;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKey& K) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        // one 32x32 -> 64-bit product each gives both halves
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k0[i], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ K.k1[i],
                       (uint32_t)p0);
    }
    return c;
}

// N counters under one key, round by round: the N chains are independent
// (their multiplies overlap) and share the key schedule, which is advanced in
// place instead of being kept as twenty round keys.
template <int N>
__device__ __forceinline__ void philox4x32_10_xn(uint4 (&c)[N], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const uint64_t p0 = (uint64_t)0xD2511F53u * c[j].x;
            const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[j].z;
            c[j] = make_uint4((uint32_t)(p1 >> 32) ^ c[j].y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c[j].w ^ k1,
                              (uint32_t)p0);
        }
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

__device__ __forceinline__ void philox4x32_10_x4(uint4 (&c)[4], uint32_t k0, uint32_t k1) {
    philox4x32_10_xn<4>(c, k0, k1);
}

enum Purpose : uint32_t { kDraftGumbel = 0, kAccept = 1, kResidualGumbel = 2, kBonusGumbel = 3 };

__device__ __forceinline__ uint32_t ctr_word3(uint32_t cycle, uint32_t purpose) {
    return (cycle << 4) | purpose;
}

// ((x >> 9) + 0.5) * 2^-23, exactly: the top 23 bits become the mantissa of a
// float in [1, 2); subtracting 1 is exact (both in [1, 2)), and adding 2^-24
// to a multiple of 2^-23 below 1 needs at most 24 significant bits.
__device__ __forceinline__ float uniform_from_bits(uint32_t x) {
    const float f = __uint_as_float((x >> 9) | 0x3F800000u);
    return __fadd_rn(__fsub_rn(f, 1.0f), 0x1p-24f);
}

// Standard Gumbel noise -log(-log u), with CUDA's accurate logf (no fast math).
__device__ __forceinline__ float gumbel_from_uniform(float u) {
    return -logf(-logf(u));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float load_elem(const void* base, int dtype, size_t idx) {
    return dtype == DSPARK_F32 ? __ldg((const float*)base + idx)
                               : bf16_bits_to_float(__ldg((const uint16_t*)base + idx));
}

// First device error wins.
__device__ __forceinline__ void report(int32_t* dev_status, int code) {
    if (dev_status) atomicCAS(dev_status, 0, code);
}

// Bounds checks of a DSPARK_DEBUG build: IN_BOUNDS(cond, status) is cond, and
// reports DSPARK_ERR_BOUNDS when cond fails, so that the guarded access can be
// skipped instead of faulting; in a normal build it is `true` and costs nothing.
// The checks cover indices computed inside the kernels (decoded tokens, rows
// of the packed target, statistics and workspace slots, pages); the inputs the
// pages define (token ids < V, cu_seqlens monotone, l <= gamma) are checked in
// every build.
#ifdef DSPARK_DEBUG
__device__ __forceinline__ bool in_bounds_check(bool cond, int32_t* dev_status) {
    if (!cond) report(dev_status, DSPARK_ERR_BOUNDS);
    return cond;
}
#define IN_BOUNDS(cond, dev_status) in_bounds_check((cond), (dev_status))
#else
#define IN_BOUNDS(cond, dev_status) true
#endif

// ---------------------------------------------------------------------------
// Reductions.
// ---------------------------------------------------------------------------
// (max, sum of exp(x - max)) pairs, merged.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 > m) {
        s = s * expf(m - m2) + s2;  // expf(-inf) = 0 covers an empty side
        m = m2;
    } else if (m2 != -INFINITY) {
        s = s + s2 * expf(m2 - m);
    }
}

// (score, index) with the larger score winning and the lower index breaking ties.
__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

template <typename T>
__device__ __forceinline__ T shfl_xor(T v, int m) {
    return __shfl_xor_sync(0xFFFFFFFFu, v, m);
}

// Global-time based bound for device spin waits (nanoseconds).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace dspark

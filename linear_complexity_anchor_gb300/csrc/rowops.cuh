// Per-row arithmetic of the tensor-core kernels in which one thread holds one token's row of
// 64 anchor scores (read from tensor memory): the row softmax over the anchors and the row
// dot product of two such rows.  The dependency chains are kept short - eight independent
// maximum chains, paired fp32 arithmetic and four partial sums, each combined in a fixed
// order - because a row warp's latency, not the multi-function unit's rate, sets how fast a
// tile's rows go (two or four row warps share a sub-partition).
#pragma once

#include <math.h>

#include "ptx.cuh"

namespace anchor {
namespace rowops {

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// In place: v_j <- 2^(c v_j - max_l c v_l) for j < m, 0 for j >= m (m >= 1); returns the sum of
// the new v_j.  c = scale * log2(e) may have either sign.  N = 64 or 128 entries per row.
template <int N>
__device__ __forceinline__ float softmax_unnormalised(float (&v)[N], int m, float c) {
    using namespace ptx;
    static_assert(N % 64 == 0, "rows of 64 or 128 entries");
    const uint64_t c2 = f32x2(c, c);
#pragma unroll
    for (int j = 0; j < N; j += 2) f32x2_split(mul_f32x2(f32x2(v[j], v[j + 1]), c2), v[j], v[j + 1]);
    if (m < N) {
#pragma unroll
        for (int j = 0; j < N; ++j)
            if (j >= m) v[j] = -INFINITY;
    }
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = max3_f32(v[i], v[i + 8], v[i + 16]);
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = max3_f32(mx8[i], v[i + 24], v[i + 32]);
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = max3_f32(mx8[i], v[i + 40], v[i + 48]);
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], v[i + 56]);
#pragma unroll
    for (int j = 64; j < N; j += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = max3_f32(mx8[i], v[j + i], v[j + 8 + i]);
    const float mx = fmaxf(max3_f32(mx8[0], mx8[1], mx8[2]), max3_f32(mx8[3], mx8[4], fmaxf(mx8[5], fmaxf(mx8[6], mx8[7]))));
    const uint64_t nb2 = f32x2(-mx, -mx);
    uint64_t z4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        float a, b;
        f32x2_split(add_f32x2(f32x2(v[j], v[j + 1]), nb2), a, b);
        a = ex2_approx(a);
        b = ex2_approx(b);
        v[j] = a;
        v[j + 1] = b;
        z4[(j >> 1) & 3] = add_f32x2(z4[(j >> 1) & 3], f32x2(a, b));
    }
    float za, zb;
    f32x2_split(add_f32x2(add_f32x2(z4[0], z4[1]), add_f32x2(z4[2], z4[3])), za, zb);
    return za + zb;
}
__device__ __forceinline__ float softmax64_unnormalised(float (&v)[64], int m, float c) {
    return softmax_unnormalised<64>(v, m, c);
}

// In place: v_j <- v_j * r (paired)
template <int N>
__device__ __forceinline__ void scale_row(float (&v)[N], float r) {
    using namespace ptx;
    const uint64_t r2 = f32x2(r, r);
#pragma unroll
    for (int j = 0; j < N; j += 2) f32x2_split(mul_f32x2(f32x2(v[j], v[j + 1]), r2), v[j], v[j + 1]);
}
__device__ __forceinline__ void scale64(float (&v)[64], float r) { scale_row<64>(v, r); }

// sum_j a_j b_j over 64 entries, as four interleaved partial sums combined in a fixed order
__device__ __forceinline__ float dot64(const float (&a)[64], const float (&b)[64]) {
    using namespace ptx;
    uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < 64; j += 2)
        s4[(j >> 1) & 3] = fma_f32x2(f32x2(a[j], a[j + 1]), f32x2(b[j], b[j + 1]), s4[(j >> 1) & 3]);
    float x, y;
    f32x2_split(add_f32x2(add_f32x2(s4[0], s4[1]), add_f32x2(s4[2], s4[3])), x, y);
    return x + y;
}

}  // namespace rowops
}  // namespace anchor

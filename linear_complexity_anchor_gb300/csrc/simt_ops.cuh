// Building blocks of the CUDA-core (fp32 FMA) kernels, shared by the forward (simt.cu) and
// the backward (backward.cu): cp.async staging of row tiles, and register-tiled contractions
// that keep one accumulator per output and add its terms in ascending index order, so that
// results are bit-identical from run to run.
#pragma once

#include "common.cuh"

#include <math.h>

namespace anchor {
namespace simt {

static __device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

static __device__ __forceinline__ uint64_t globaltimer_now() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 16-byte asynchronous copy global -> shared (cached in L2 only)
static __device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
static __device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> static __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows x d elements of a row-major [rows][d] global matrix into shared memory with a row pitch
// of `pitch` elements; every row is a whole number of 16-byte pieces (d * sizeof(T) >= 32)
template <typename T>
static __device__ __forceinline__ void stage_rows(T *dst, const T *__restrict__ src, int rows, int d, int pitch) {
    const int per_row = d * (int)sizeof(T) / 16;
    for (int c = threadIdx.x; c < rows * per_row; c += blockDim.x) {
        const int r = c / per_row, k = c - r * per_row;
        cp_async16(reinterpret_cast<char *>(dst + (size_t)r * pitch) + 16 * k,
                   reinterpret_cast<const char *>(src + (size_t)r * d) + 16 * k);
    }
}

// four consecutive elements as floats (bf16 widens exactly)
static __device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
static __device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}

// eight outputs of one row to global memory: 16 bytes of bf16 or 32 bytes of fp32
static __device__ __forceinline__ void st8(float *dst, const float *v) {
    reinterpret_cast<float4 *>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
static __device__ __forceinline__ void st8(__nv_bfloat16 *dst, const float *v) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}

// As[r][j] = scale * sum_k Qs[r][k] Us[j][k] (k ascending), r < rows, j < m.  Each thread
// takes 4 x 4 outputs: rows rt + a nrt and anchors ct + b nct (a, b < 4), so that lanes,
// which take consecutive ct, read consecutive U rows (distinct banks) and share Q rows.
template <typename T>
static __device__ __forceinline__ void scores(const T *Qs, const T *Us, int pitch, float *As, int ap, int rows, int m, int d,
                                       float scale) {
    const int nct = (m + 3) / 4, nrt = (rows + 3) / 4;
    for (int t = threadIdx.x; t < nrt * nct; t += blockDim.x) {
        const int rt = t / nct, ct = t - rt * nct;
        const T *q[4], *u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[i] = Qs + (size_t)min(rt + i * nrt, rows - 1) * pitch;
            u[i] = Us + (size_t)min(ct + i * nct, m - 1) * pitch;
        }
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
        for (int k = 0; k < d; k += 4) {
            float4 qa[4], ua[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qa[i] = ld4(q[i] + k);
                ua[i] = ld4(u[i] + k);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float s = acc[a][b];
                    s = __fmaf_rn(qa[a].x, ua[b].x, s);
                    s = __fmaf_rn(qa[a].y, ua[b].y, s);
                    s = __fmaf_rn(qa[a].z, ua[b].z, s);
                    acc[a][b] = __fmaf_rn(qa[a].w, ua[b].w, s);
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int r = rt + a * nrt, j = ct + b * nct;
                if (r < rows && j < m) As[(size_t)r * ap + j] = __fmul_rn(scale, acc[a][b]);
            }
    }
}

// scores() for an As laid over Qs: each thread first computes its (at most two) 4 x 4 tiles
// into registers, then every thread of the CTA meets (all have read Qs), then the tiles are
// written.  The same sums in the same order as scores().  Needs ceil(rows / 4) ceil(m / 4)
// <= 2 blockDim.x; every thread of the CTA must call it.
template <typename T>
static __device__ __forceinline__ void scores_over(const T *Qs, const T *Us, int pitch, float *As, int ap, int rows, int m,
                                                   int d, float scale) {
    const int nct = (m + 3) / 4, nrt = (rows + 3) / 4;
    float acc[2][4][4];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int t = threadIdx.x + it * blockDim.x;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[it][a][b] = 0.f;
        if (t >= nrt * nct) continue;
        const int rt = t / nct, ct = t - rt * nct;
        const T *q[4], *u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[i] = Qs + (size_t)min(rt + i * nrt, rows - 1) * pitch;
            u[i] = Us + (size_t)min(ct + i * nct, m - 1) * pitch;
        }
        for (int k = 0; k < d; k += 4) {
            float4 qa[4], ua[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qa[i] = ld4(q[i] + k);
                ua[i] = ld4(u[i] + k);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float s = acc[it][a][b];
                    s = __fmaf_rn(qa[a].x, ua[b].x, s);
                    s = __fmaf_rn(qa[a].y, ua[b].y, s);
                    s = __fmaf_rn(qa[a].z, ua[b].z, s);
                    acc[it][a][b] = __fmaf_rn(qa[a].w, ua[b].w, s);
                }
        }
    }
    __syncthreads();  // Qs is read: As may overwrite it
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int t = threadIdx.x + it * blockDim.x;
        if (t >= nrt * nct) continue;
        const int rt = t / nct, ct = t - rt * nct;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int r = rt + a * nrt, j = ct + b * nct;
                if (r < rows && j < m) As[(size_t)r * ap + j] = __fmul_rn(scale, acc[it][a][b]);
            }
    }
}

// Row softmax of As in place, one thread per row: A_ij = exp(S_ij - max_j S_ij) * (1 / sum).
static __device__ __forceinline__ void softmax_rows(float *As, int ap, int rows, int m) {
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        float *a = As + (size_t)r * ap;
        float mx = -INFINITY;
#pragma unroll 4
        for (int j = 0; j < m; ++j) mx = fmaxf(mx, a[j]);
        float z = 0.f;
#pragma unroll 4
        for (int j = 0; j < m; ++j) {
            const float e = expf(__fsub_rn(a[j], mx));
            a[j] = e;
            z = __fadd_rn(z, e);
        }
        const float rz = __frcp_rn(z);
#pragma unroll 4
        for (int j = 0; j < m; ++j) a[j] = __fmul_rn(a[j], rz);
    }
}

// Wacc[j][k] += sum_r As[r][j] Vs[r][k] and Dacc[j] += sum_r As[r][j] (r ascending).  Each
// thread takes 2 anchors x 4 columns; lanes of a warp take consecutive columns; the threads of
// column block 0 also sum the two anchors' Delta from the A values they already hold.
template <typename T>
static __device__ __forceinline__ void accumulate(const float *As, int ap, const T *Vs, int pitch, float *Wacc, float *Dacc,
                                           int rows, int m, int d) {
    const int nct = d / 4, njt = (m + 1) / 2;
    for (int t = threadIdx.x; t < njt * nct; t += blockDim.x) {
        const int jt = t / nct, ct = t - jt * nct;
        const int j0 = jt * 2, k0 = ct * 4;
        const bool two = j0 + 1 < m;
        float4 w0 = *reinterpret_cast<const float4 *>(Wacc + (size_t)j0 * d + k0);
        float4 w1 = two ? *reinterpret_cast<const float4 *>(Wacc + (size_t)(j0 + 1) * d + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
        const bool delta = Dacc != nullptr && ct == 0;
        float d0 = delta ? Dacc[j0] : 0.f, d1 = delta && two ? Dacc[j0 + 1] : 0.f;
        const float *a = As + j0;
        const int j1 = two ? 1 : 0;
#pragma unroll 4
        for (int r = 0; r < rows; ++r) {
            const float a0 = a[(size_t)r * ap], a1 = a[(size_t)r * ap + j1];
            const float4 v = ld4(Vs + (size_t)r * pitch + k0);
            w0.x = __fmaf_rn(a0, v.x, w0.x);
            w0.y = __fmaf_rn(a0, v.y, w0.y);
            w0.z = __fmaf_rn(a0, v.z, w0.z);
            w0.w = __fmaf_rn(a0, v.w, w0.w);
            w1.x = __fmaf_rn(a1, v.x, w1.x);
            w1.y = __fmaf_rn(a1, v.y, w1.y);
            w1.z = __fmaf_rn(a1, v.z, w1.z);
            w1.w = __fmaf_rn(a1, v.w, w1.w);
            d0 = __fadd_rn(d0, a0);
            d1 = __fadd_rn(d1, a1);
        }
        *reinterpret_cast<float4 *>(Wacc + (size_t)j0 * d + k0) = w0;
        if (two) *reinterpret_cast<float4 *>(Wacc + (size_t)(j0 + 1) * d + k0) = w1;
        if (delta) {
            Dacc[j0] = d0;
            if (two) Dacc[j0 + 1] = d1;
        }
    }
}

// W'[j][k] = W[j][k] / Delta_j in place (0 where Delta_j = 0: an anchor no token reaches)
static __device__ __forceinline__ void normalise(float *W, const float *Dl, int m, int d) {
    for (int p = threadIdx.x; p < m * d; p += blockDim.x) {
        const float dj = Dl[p / d];
        W[p] = dj != 0.f ? __fdiv_rn(W[p], dj) : 0.f;
    }
}

// eight consecutive values of a shared-memory row as floats
static __device__ __forceinline__ void ld8(const float *p, float *w) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
}
static __device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float *w) {
    const float4 a = ld4(p), b = ld4(p + 4);
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
}

// Hg[r][k] = post * sum_j As[r][j] Ws[j][k] (j ascending) for r < rows, stored to the global
// rows at Hg (row-major, d columns); Ws rows have `wpitch` elements (float, or the input
// type).  Each thread takes 2 rows x 8 columns (one 16-byte bf16 store, or two fp32 ones, per
// row); lanes of a warp take consecutive columns.
template <typename T, typename TW>
static __device__ __forceinline__ void apply(const float *As, int ap, const TW *Ws, int wpitch, T *__restrict__ Hg,
                                             int rows, int m, int d, float post) {
    const int nct = d / 8, nrt = (rows + 1) / 2;
    for (int t = threadIdx.x; t < nrt * nct; t += blockDim.x) {
        const int rt = t / nct, ct = t - rt * nct;
        const int r0 = rt * 2, k0 = ct * 8;
        const bool two = r0 + 1 < rows;
        const float *a0 = As + (size_t)r0 * ap, *a1 = As + (size_t)(two ? r0 + 1 : r0) * ap;
        float acc[2][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[0][c] = acc[1][c] = 0.f;
#pragma unroll 4
        for (int j = 0; j < m; ++j) {
            const float x0 = a0[j], x1 = a1[j];
            float w[8];
            ld8(Ws + (size_t)j * wpitch + k0, w);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                acc[0][c] = __fmaf_rn(x0, w[c], acc[0][c]);
                acc[1][c] = __fmaf_rn(x1, w[c], acc[1][c]);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            acc[0][c] = __fmul_rn(post, acc[0][c]);
            acc[1][c] = __fmul_rn(post, acc[1][c]);
        }
        st8(Hg + (size_t)r0 * d + k0, acc[0]);
        if (two) st8(Hg + (size_t)(r0 + 1) * d + k0, acc[1]);
    }
}

template <typename T> constexpr int pad_elems() { return 16 / (int)sizeof(T); }

}  // namespace simt
}  // namespace anchor

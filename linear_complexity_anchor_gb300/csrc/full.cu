// Approximation-error diagnostic of the anchor construction: full softmax attention,
//   H_full[i] = sum_j softmax over j of (scale q_i . k_j) v_j,
// the quadratic construction the anchors approximate, and the per-slice relative Frobenius
// error ||H_full - H_anchor||_F / ||H_full||_F (the skeptic's concrete test in the
// pith.science verdict on arXiv 2505.16463: anchors taken from rows of the keys).
//
// full_attn_kernel: one CTA per 64 queries of a slice; the keys and values stream through in
// 64-row tiles (cp.async), with the running row maximum, row sum and output rescaled tile by
// tile (online softmax).  The tiles are visited in order and every sum is taken in a fixed
// order, so results are bit-identical from run to run.  CUDA-core fp32 arithmetic; used for
// the diagnostic, not on the anchor path.
// rel_error_kernel: one CTA per slice, fixed-order partial sums then a fixed tree.
#include "common.cuh"
#include "simt_ops.cuh"

#include <math.h>

namespace anchor {
namespace {

using namespace simt;

constexpr int kThreads = 256;
constexpr int kQT = 64;  // queries per CTA
constexpr int kKT = 64;  // keys per tile

template <typename T> size_t full_smem(int d) {
    const size_t pitch = d + pad_elems<T>();
    return sizeof(T) * 3 * (size_t)kQT * pitch + 4 * ((size_t)kQT * (kKT + 1) + (size_t)kQT * d + 3 * kQT);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
full_attn_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V, T *__restrict__ H,
                 int heads, int n, int d, float scale) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int pitch = d + pad_elems<T>();
    const int ap = kKT + 1;
    T *Qs = reinterpret_cast<T *>(smem);                   // [kQT][pitch]
    T *Ks = Qs + (size_t)kQT * pitch;                      // [kKT][pitch]
    T *Vs = Ks + (size_t)kKT * pitch;                      // [kKT][pitch]
    float *Ps = reinterpret_cast<float *>(Vs + (size_t)kKT * pitch);  // [kQT][ap] scores, then weights
    float *O = Ps + (size_t)kQT * ap;                      // [kQT][d] running output
    float *mrow = O + (size_t)kQT * d, *lrow = mrow + kQT, *corr = lrow + kQT;
    const long long slice = blockIdx.y;
    const int h = (int)(slice % heads);
    const int q0 = blockIdx.x * kQT, rows = min(kQT, n - q0);
    const size_t off = (size_t)slice * n * d;
    const T *Kh = K + (size_t)h * n * d;

    stage_rows(Qs, Q + off + (size_t)q0 * d, rows, d, pitch);
    cp_async_commit();
    for (int i = threadIdx.x; i < kQT * d; i += blockDim.x) O[i] = 0.f;
    for (int r = threadIdx.x; r < kQT; r += blockDim.x) {
        mrow[r] = -INFINITY;
        lrow[r] = 0.f;
    }
    for (int j0 = 0; j0 < n; j0 += kKT) {
        const int kr = min(kKT, n - j0);
        __syncthreads();  // the last tile's Ks, Vs and Ps are read
        stage_rows(Ks, Kh + (size_t)j0 * d, kr, d, pitch);
        stage_rows(Vs, V + off + (size_t)j0 * d, kr, d, pitch);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        scores(Qs, Ks, pitch, Ps, ap, rows, kr, d, scale);
        __syncthreads();
        // online softmax, one thread per query row: new maximum, weights of this tile, the
        // factor that rescales the row's running sum and output
        for (int r = threadIdx.x; r < rows; r += blockDim.x) {
            float *p = Ps + (size_t)r * ap;
            float mx = mrow[r];
            for (int j = 0; j < kr; ++j) mx = fmaxf(mx, p[j]);
            const float c = expf(__fsub_rn(mrow[r], mx));  // 0 on the first tile (exp(-inf))
            float z = 0.f;
            for (int j = 0; j < kr; ++j) {
                const float e = expf(__fsub_rn(p[j], mx));
                p[j] = e;
                z = __fadd_rn(z, e);
            }
            lrow[r] = __fmaf_rn(lrow[r], c, z);
            mrow[r] = mx;
            corr[r] = c;
        }
        __syncthreads();
        // O[r][k] = O[r][k] corr_r + sum_j P[r][j] V[j][k] (j ascending); 2 rows x 4 columns
        const int nct = d / 4, nrt = (rows + 1) / 2;
        for (int t = threadIdx.x; t < nrt * nct; t += blockDim.x) {
            const int rt = t / nct, ct = t - rt * nct;
            const int r0 = rt * 2, k0 = ct * 4;
            const bool two = r0 + 1 < rows;
            float4 a = *reinterpret_cast<float4 *>(O + (size_t)r0 * d + k0);
            float4 b = two ? *reinterpret_cast<float4 *>(O + (size_t)(r0 + 1) * d + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float c0 = corr[r0], c1 = two ? corr[r0 + 1] : 0.f;
            a = make_float4(__fmul_rn(a.x, c0), __fmul_rn(a.y, c0), __fmul_rn(a.z, c0), __fmul_rn(a.w, c0));
            b = make_float4(__fmul_rn(b.x, c1), __fmul_rn(b.y, c1), __fmul_rn(b.z, c1), __fmul_rn(b.w, c1));
            const float *p0 = Ps + (size_t)r0 * ap, *p1 = Ps + (size_t)(two ? r0 + 1 : r0) * ap;
            for (int j = 0; j < kr; ++j) {
                const float4 v = ld4(Vs + (size_t)j * pitch + k0);
                const float x0 = p0[j], x1 = p1[j];
                a.x = __fmaf_rn(x0, v.x, a.x);
                a.y = __fmaf_rn(x0, v.y, a.y);
                a.z = __fmaf_rn(x0, v.z, a.z);
                a.w = __fmaf_rn(x0, v.w, a.w);
                b.x = __fmaf_rn(x1, v.x, b.x);
                b.y = __fmaf_rn(x1, v.y, b.y);
                b.z = __fmaf_rn(x1, v.z, b.z);
                b.w = __fmaf_rn(x1, v.w, b.w);
            }
            *reinterpret_cast<float4 *>(O + (size_t)r0 * d + k0) = a;
            if (two) *reinterpret_cast<float4 *>(O + (size_t)(r0 + 1) * d + k0) = b;
        }
    }
    __syncthreads();
    // H = O / l, 8 columns per thread (16-byte bf16 or two fp32 stores)
    const int nct = d / 8;
    for (int t = threadIdx.x; t < rows * nct; t += blockDim.x) {
        const int r = t / nct, k0 = (t - r * nct) * 8;
        float v[8];
        for (int c = 0; c < 8; ++c) v[c] = __fdiv_rn(O[(size_t)r * d + k0 + c], lrow[r]);
        st8(H + off + (size_t)(q0 + r) * d + k0, v);
    }
}

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(kThreads)
rel_error_kernel(const T *__restrict__ Href, const T *__restrict__ H, float *__restrict__ err, size_t per_slice) {
    __shared__ float s_num[kThreads], s_den[kThreads];
    const size_t off = (size_t)blockIdx.x * per_slice;
    float num = 0.f, den = 0.f;
    for (size_t e = threadIdx.x; e < per_slice; e += blockDim.x) {
        const float a = widen(Href[off + e]), b = widen(H[off + e]);
        const float dlt = __fsub_rn(a, b);
        num = __fmaf_rn(dlt, dlt, num);
        den = __fmaf_rn(a, a, den);
    }
    s_num[threadIdx.x] = num;
    s_den[threadIdx.x] = den;
    for (int w = kThreads / 2; w > 0; w >>= 1) {
        __syncthreads();
        if (threadIdx.x < w) {
            s_num[threadIdx.x] = __fadd_rn(s_num[threadIdx.x], s_num[threadIdx.x + w]);
            s_den[threadIdx.x] = __fadd_rn(s_den[threadIdx.x], s_den[threadIdx.x + w]);
        }
    }
    if (threadIdx.x == 0) err[blockIdx.x] = s_den[0] > 0.f ? sqrtf(s_num[0]) / sqrtf(s_den[0]) : 0.f;
}

template <typename T>
cudaError_t full_launch_t(const FullProblem &p, cudaStream_t stream) {
    const size_t smem = full_smem<T>(p.d);
    cudaError_t e = cudaFuncSetAttribute(full_attn_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((p.n + kQT - 1) / kQT), (unsigned)p.slices());
    full_attn_kernel<T><<<grid, kThreads, smem, stream>>>((const T *)p.Q, (const T *)p.K, (const T *)p.V, (T *)p.H,
                                                         p.heads, p.n, p.d, p.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_full_attention(const FullProblem &p, cudaStream_t stream) {
    return p.f32 ? full_launch_t<float>(p, stream) : full_launch_t<__nv_bfloat16>(p, stream);
}

cudaError_t launch_rel_error(const void *Href, const void *H, float *err, long long slices, size_t per_slice, bool f32,
                             cudaStream_t stream) {
    if (f32)
        rel_error_kernel<float><<<(unsigned)slices, kThreads, 0, stream>>>((const float *)Href, (const float *)H, err,
                                                                          per_slice);
    else
        rel_error_kernel<__nv_bfloat16><<<(unsigned)slices, kThreads, 0, stream>>>(
            (const __nv_bfloat16 *)Href, (const __nv_bfloat16 *)H, err, per_slice);
    return cudaGetLastError();
}

}  // namespace anchor

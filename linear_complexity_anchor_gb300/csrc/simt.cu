// CUDA-core (fp32 FMA) variants of the anchor-attention forward
//   H = A Delta^{-1} (A^T V),  A = rowsoftmax(scale * Q U^T),  Delta = diag(colsum A)
// (AnchorFormer, arXiv 2505.16463; pith.science verdict, "key_machinery" and the referee
// summary of Eq. 11/12).  Used for the fp32 entry point, for m < 32 (where a tensor-core
// tile would be mostly padding) and for shapes the tensor-core path does not cover.
//
// Two variants:
//   slice : one CTA holds a whole (batch, head) slice in shared memory and runs every step
//           (scores, softmax, Delta, A^T V, Delta^{-1}, A W').  No workspace.
//   split : the n tokens of a slice are cut into fixed 512-token chunks.  Kernel 1 gives
//           each chunk's partial (Delta, A^T V); kernel 2 sums the partials of a slice in
//           chunk order and divides by Delta; kernel 3 recomputes A tile by tile with the
//           same code as kernel 1 and forms H = A W'.  The chunk count depends on n only,
//           so the summation order - and the result - is fixed.
#include "common.cuh"

#include <math.h>

namespace anchor {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// rows x d elements of a row-major global matrix into shared memory with row pitch `pitch`.
template <typename T>
__device__ __forceinline__ void load_rows(const T *__restrict__ src, float *dst, int rows, int d,
                                          int pitch) {
    const int count = rows * d;
    for (int e = threadIdx.x; e < count; e += blockDim.x) {
        const int r = e / d;
        dst[r * pitch + (e - r * d)] = to_f32(src[e]);
    }
}

// As[r][j] = softmax_j(scale * Xs[r] . Us[j]) for r < rows.  Called by the whole CTA; the
// caller synchronises before (Xs, Us ready) and after (As ready).
__device__ __forceinline__ void scores_softmax(const float *Xs, const float *Us, float *As, int rows,
                                               int m, int d, int dp, int mp, float scale) {
    for (int p = threadIdx.x; p < rows * m; p += blockDim.x) {
        const int r = p / m;
        const int j = p - r * m;
        const float *q = Xs + r * dp;
        const float *u = Us + j * dp;
        float s = 0.f;
        for (int k = 0; k < d; ++k) s = __fmaf_rn(q[k], u[k], s);
        As[r * mp + j] = __fmul_rn(scale, s);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = warp; r < rows; r += kWarps) {
        float *a = As + r * mp;
        float mx = -INFINITY;
        for (int j = lane; j < m; j += 32) mx = fmaxf(mx, a[j]);
        mx = warp_max(mx);
        float z = 0.f;
        for (int j = lane; j < m; j += 32) {
            const float e = expf(__fsub_rn(a[j], mx));
            a[j] = e;
            z = __fadd_rn(z, e);
        }
        z = warp_sum(z);
        for (int j = lane; j < m; j += 32) a[j] = __fdiv_rn(a[j], z);
    }
}

// ------------------------------------------------------------------ whole slice per CTA
template <typename T>
__global__ void __launch_bounds__(kThreads)
simt_slice_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V,
                  T *__restrict__ H, int heads, int n, int m, int d, float scale) {
    extern __shared__ float sm[];
    const int dp = d + 1, mp = m + 1;
    float *Us = sm;             // [m][dp]
    float *Xs = Us + m * dp;    // [n][dp]  Q, then V
    float *As = Xs + n * dp;    // [n][mp]
    float *Ws = As + n * mp;    // [m][d]   W' = Delta^{-1} A^T V
    float *Ds = Ws + m * d;     // [m]      Delta
    const long long slice = blockIdx.x;
    const int h = (int)(slice % heads);
    const size_t off = (size_t)slice * n * d;

    load_rows(U + (size_t)h * m * d, Us, m, d, dp);
    load_rows(Q + off, Xs, n, d, dp);
    __syncthreads();
    scores_softmax(Xs, Us, As, n, m, d, dp, mp, scale);
    __syncthreads();
    load_rows(V + off, Xs, n, d, dp);
    for (int j = threadIdx.x; j < m; j += blockDim.x) {
        float s = 0.f;
        for (int i = 0; i < n; ++i) s = __fadd_rn(s, As[i * mp + j]);
        Ds[j] = s;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < m * d; p += blockDim.x) {
        const int j = p / d, k = p - j * d;
        float s = 0.f;
        for (int i = 0; i < n; ++i) s = __fmaf_rn(As[i * mp + j], Xs[i * dp + k], s);
        Ws[p] = Ds[j] != 0.f ? __fdiv_rn(s, Ds[j]) : 0.f;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < n * d; p += blockDim.x) {
        const int i = p / d, k = p - i * d;
        float s = 0.f;
        for (int j = 0; j < m; ++j) s = __fmaf_rn(As[i * mp + j], Ws[j * d + k], s);
        H[off + p] = from_f32<T>(s);
    }
}

// ------------------------------------------------------------------ split variant
// Partial of chunk c of a slice: Delta_c[j] = sum_{i in c} A_ij and W_c[j][k] =
// sum_{i in c} A_ij V_ik, written to part[(slice * splits + c) * (m*d + m)].
template <typename T>
__global__ void __launch_bounds__(kThreads)
simt_partial_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V,
                    float *__restrict__ part, int heads, int n, int m, int d, float scale,
                    int splits) {
    extern __shared__ float sm[];
    const int dp = d + 1, mp = m + 1;
    float *Us = sm;                     // [m][dp]
    float *Xs = Us + m * dp;            // [kSimtTile][dp]
    float *As = Xs + kSimtTile * dp;    // [kSimtTile][mp]
    float *Wacc = As + kSimtTile * mp;  // [m][d]
    float *Dacc = Wacc + m * d;         // [m]
    const long long slice = blockIdx.x / splits;
    const int c = (int)(blockIdx.x - slice * splits);
    const int h = (int)(slice % heads);
    const size_t off = (size_t)slice * n * d;
    const int t_begin = c * kSimtChunk;
    const int t_end = min(n, t_begin + kSimtChunk);

    load_rows(U + (size_t)h * m * d, Us, m, d, dp);
    for (int p = threadIdx.x; p < m * d + m; p += blockDim.x) Wacc[p] = 0.f;
    for (int t0 = t_begin; t0 < t_end; t0 += kSimtTile) {
        const int rows = min(kSimtTile, t_end - t0);
        __syncthreads();
        load_rows(Q + off + (size_t)t0 * d, Xs, rows, d, dp);
        __syncthreads();
        scores_softmax(Xs, Us, As, rows, m, d, dp, mp, scale);
        __syncthreads();
        load_rows(V + off + (size_t)t0 * d, Xs, rows, d, dp);
        __syncthreads();
        for (int j = threadIdx.x; j < m; j += blockDim.x) {
            float s = Dacc[j];
            for (int r = 0; r < rows; ++r) s = __fadd_rn(s, As[r * mp + j]);
            Dacc[j] = s;
        }
        for (int p = threadIdx.x; p < m * d; p += blockDim.x) {
            const int j = p / d, k = p - j * d;
            float s = Wacc[p];
            for (int r = 0; r < rows; ++r) s = __fmaf_rn(As[r * mp + j], Xs[r * dp + k], s);
            Wacc[p] = s;
        }
    }
    __syncthreads();
    float *dst = part + ((size_t)slice * splits + c) * (size_t)(m * d + m);
    for (int p = threadIdx.x; p < m * d + m; p += blockDim.x) dst[p] = Wacc[p];
}

// W'[slice] = (sum over chunks, in chunk order, of W_c) / (sum of Delta_c); 0 where Delta = 0.
__global__ void __launch_bounds__(kThreads)
simt_reduce_kernel(const float *__restrict__ part, float *__restrict__ Wp, int m, int d, int splits) {
    extern __shared__ float Ds[];  // [m]
    const long long slice = blockIdx.x;
    const size_t stride = (size_t)(m * d + m);
    const float *base = part + (size_t)slice * splits * stride;
    for (int j = threadIdx.x; j < m; j += blockDim.x) {
        float s = 0.f;
        for (int c = 0; c < splits; ++c) s = __fadd_rn(s, base[c * stride + m * d + j]);
        Ds[j] = s;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < m * d; p += blockDim.x) {
        float s = 0.f;
        for (int c = 0; c < splits; ++c) s = __fadd_rn(s, base[c * stride + p]);
        const float dj = Ds[p / d];
        Wp[(size_t)slice * m * d + p] = dj != 0.f ? __fdiv_rn(s, dj) : 0.f;
    }
}

// H rows of one kSimtTile-token tile: recompute A (same code as the partial kernel), then
// H = A W'.
template <typename T>
__global__ void __launch_bounds__(kThreads)
simt_apply_kernel(const T *__restrict__ Q, const T *__restrict__ U, const float *__restrict__ Wp,
                  T *__restrict__ H, int heads, int n, int m, int d, float scale) {
    extern __shared__ float sm[];
    const int dp = d + 1, mp = m + 1;
    float *Us = sm;                   // [m][dp]
    float *Xs = Us + m * dp;          // [kSimtTile][dp]
    float *As = Xs + kSimtTile * dp;  // [kSimtTile][mp]
    float *Ws = As + kSimtTile * mp;  // [m][d]
    const int tiles = (n + kSimtTile - 1) / kSimtTile;
    const long long slice = blockIdx.x / tiles;
    const int h = (int)(slice % heads);
    const size_t off = (size_t)slice * n * d;
    const int t0 = (int)(blockIdx.x - slice * tiles) * kSimtTile;
    const int rows = min(kSimtTile, n - t0);

    load_rows(U + (size_t)h * m * d, Us, m, d, dp);
    load_rows(Q + off + (size_t)t0 * d, Xs, rows, d, dp);
    const float *wsrc = Wp + (size_t)slice * m * d;
    for (int p = threadIdx.x; p < m * d; p += blockDim.x) Ws[p] = wsrc[p];
    __syncthreads();
    scores_softmax(Xs, Us, As, rows, m, d, dp, mp, scale);
    __syncthreads();
    T *out = H + off + (size_t)t0 * d;
    for (int p = threadIdx.x; p < rows * d; p += blockDim.x) {
        const int r = p / d, k = p - r * d;
        float s = 0.f;
        for (int j = 0; j < m; ++j) s = __fmaf_rn(As[r * mp + j], Ws[j * d + k], s);
        out[p] = from_f32<T>(s);
    }
}

template <typename T>
cudaError_t slice_launch(const Problem &p, cudaStream_t stream) {
    const size_t smem = simt_slice_smem_bytes(p.n, p.m, p.d);
    cudaError_t e = cudaFuncSetAttribute(simt_slice_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    simt_slice_kernel<T><<<(unsigned)p.slices(), kThreads, smem, stream>>>(
        (const T *)p.Q, (const T *)p.U, (const T *)p.V, (T *)p.H, p.heads, p.n, p.m, p.d, p.scale);
    return cudaGetLastError();
}

template <typename T>
cudaError_t split_launch(const Problem &p, int splits, float *ws, cudaStream_t stream) {
    const size_t smem = simt_split_smem_bytes(p.m, p.d);
    cudaError_t e = cudaFuncSetAttribute(simt_partial_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(simt_apply_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    float *part = ws;
    float *Wp = ws + (size_t)p.slices() * splits * (size_t)(p.m * p.d + p.m);
    simt_partial_kernel<T><<<(unsigned)(p.slices() * splits), kThreads, smem, stream>>>(
        (const T *)p.Q, (const T *)p.U, (const T *)p.V, part, p.heads, p.n, p.m, p.d, p.scale, splits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    simt_reduce_kernel<<<(unsigned)p.slices(), kThreads, sizeof(float) * p.m, stream>>>(part, Wp, p.m, p.d,
                                                                                       splits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const unsigned tiles = (unsigned)((p.n + kSimtTile - 1) / kSimtTile);
    simt_apply_kernel<T><<<(unsigned)(p.slices() * tiles), kThreads, smem, stream>>>(
        (const T *)p.Q, (const T *)p.U, Wp, (T *)p.H, p.heads, p.n, p.m, p.d, p.scale);
    return cudaGetLastError();
}

}  // namespace

size_t simt_slice_smem_bytes(int n, int m, int d) {
    const size_t dp = d + 1, mp = m + 1;
    return sizeof(float) * ((size_t)m * dp + (size_t)n * dp + (size_t)n * mp + (size_t)m * d + m);
}

size_t simt_split_smem_bytes(int m, int d) {
    const size_t dp = d + 1, mp = m + 1;
    // partial: Us + Xs + As + Wacc + Dacc; apply: Us + Xs + As + Ws (smaller)
    return sizeof(float) * ((size_t)m * dp + kSimtTile * dp + kSimtTile * mp + (size_t)m * d + m);
}

size_t simt_split_workspace_bytes(const Problem &p, int splits) {
    const size_t per = (size_t)p.m * p.d + p.m;
    return sizeof(float) * ((size_t)p.slices() * splits * per + (size_t)p.slices() * p.m * p.d);
}

cudaError_t launch_simt_slice(const Problem &p, cudaStream_t stream) {
    return p.f32 ? slice_launch<float>(p, stream) : slice_launch<__nv_bfloat16>(p, stream);
}

cudaError_t launch_simt_split(const Problem &p, int splits, float *workspace, cudaStream_t stream) {
    return p.f32 ? split_launch<float>(p, splits, workspace, stream)
                 : split_launch<__nv_bfloat16>(p, splits, workspace, stream);
}

}  // namespace anchor

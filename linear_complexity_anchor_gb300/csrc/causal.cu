// Masked (causal) variant of the anchor-attention forward: the anchors' summaries seen by
// token i include only tokens j <= i, so that no token draws on a later one (one of the
// inferences of the pith.science verdict on arXiv 2505.16463: A can be masked against later
// tokens without giving up the O(mn) cost):
//   Delta^(i)_l = sum_{j<=i} A[j][l],  W^(i)_l = sum_{j<=i} A[j][l] v_j,
//   H[i] = sum_l A[i][l] W^(i)_l / Delta^(i)_l   (0 for an anchor with Delta^(i)_l = 0).
//
// A chunked scan on CUDA cores (fp32 FMA), one launch, work items from a ticket in a fixed
// order: every C1 item (a 512-token chunk: its totals Delta_c, A^T V), then every C2 item.
// The last C1 chunk of a slice to finish writes each chunk's exclusive prefix (the sums of
// the chunks before it, in chunk order).  A C2 item starts from its chunk's prefix (W, Delta)
// and walks the chunk in tiles of TR tokens: with B[i][l] = A[i][l] / Delta^(i)_l (Delta^(i)
// running down the tile from the prefix),
//   H_tile = B W + mask_{j<=i}(B A_tile^T) V_tile,
// then adds the tile to the prefix.  So the work is O(n m d + n TR (m + d)) per slice, every
// sum is taken in a fixed order, and results are bit-identical from run to run.
#include "common.cuh"
#include "simt_ops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_causal_error;  // bit 1: a wait for a slice's prefixes gave up

namespace {

using namespace simt;

constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;

__host__ __device__ __forceinline__ int pad4(int m) { return (m + 3) & ~3; }
// floats per chunk of the prefix array: W [m][d] | Delta [m, padded]: read with 16-byte copies
__host__ __device__ __forceinline__ size_t pre_stride(int m, int d) { return (size_t)m * d + pad4(m); }

struct CausalParams {
    int heads, n, m, d;
    float scale;
    int slices, chunks, tile;
    unsigned *ticket, *arrived, *ready;
    float *part;  // [slices][chunks][m + m d]  Delta_c | (A^T V)_c
    float *pre;   // [slices][chunks][m d + m4] the sums of the chunks before c
    uint64_t wait_ns;
};

// Us [m][pitch] | Qs, Vs [TR][pitch] (input type) | W [m][d] | Dl [m4] | Ht [TR][d] | As, Bs
// [TR][m+1] | Cs [TR][TR+1] (fp32)
template <typename T> size_t causal_smem(int m, int d, int tile) {
    const size_t pitch = d + pad_elems<T>();
    return sizeof(T) * ((size_t)m + 2 * tile) * pitch +
           4 * ((size_t)m * d + pad4(m) + (size_t)tile * d + 2 * (size_t)tile * (m + 1) + (size_t)tile * (tile + 1));
}

template <typename T> int causal_tile(int m, int d) {
    for (int tile = 64; tile >= 8; tile /= 2)
        if (causal_smem<T>(m, d, tile) <= kSimtMaxSmem) return tile;
    return 0;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
causal_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V, T *__restrict__ H,
              const CausalParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ unsigned s_item;
    __shared__ int s_flag;
    const int m = p.m, d = p.d, TR = p.tile;
    const int pitch = d + pad_elems<T>();
    const int ap = m + 1, cp = TR + 1;
    T *Us = reinterpret_cast<T *>(smem);
    T *Qs = Us + (size_t)m * pitch;
    T *Vs = Qs + (size_t)TR * pitch;
    float *W = reinterpret_cast<float *>(Vs + (size_t)TR * pitch);
    float *Dl = W + (size_t)m * d;
    float *Ht = Dl + pad4(m);
    float *As = Ht + (size_t)TR * d;
    float *Bs = As + (size_t)TR * ap;
    float *Cs = Bs + (size_t)TR * ap;
    const unsigned n1 = (unsigned)(p.slices * p.chunks);
    const size_t md = (size_t)m * d;
    const size_t pst = (size_t)m + md;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_item = atomicAdd(p.ticket, 1u);
        __syncthreads();
        const unsigned item = s_item;
        if (item >= 2 * n1) break;
        const bool c1 = item < n1;
        const unsigned it = c1 ? item : item - n1;
        const int slice = (int)(it / p.chunks), c = (int)(it % p.chunks);
        const int h = slice % p.heads;
        const size_t off = (size_t)slice * p.n * d;
        const int t_begin = c * kSimtChunk, t_end = min(p.n, t_begin + kSimtChunk);
        stage_rows(Us, U + (size_t)h * md, m, d, pitch);
        if (c1) {
            // ------------------------------------------------ C1: the chunk's totals
            cp_async_commit();
            for (int i = threadIdx.x; i < (int)md; i += blockDim.x) W[i] = 0.f;
            for (int i = threadIdx.x; i < m; i += blockDim.x) Dl[i] = 0.f;
            for (int t0 = t_begin; t0 < t_end; t0 += TR) {
                const int rows = min(TR, t_end - t0);
                __syncthreads();
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Vs, V + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                accumulate(As, ap, Vs, pitch, W, Dl, rows, m, d);
            }
            __syncthreads();
            float *dst = p.part + ((size_t)slice * p.chunks + c) * pst;
            for (int i = threadIdx.x; i < m; i += blockDim.x) dst[i] = Dl[i];
            for (int i = threadIdx.x; i < (int)md; i += blockDim.x) dst[m + i] = W[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_flag = atomicAdd(p.arrived + slice, 1u) == (unsigned)(p.chunks - 1);
            __syncthreads();
            if (!s_flag) continue;
            // the last chunk of the slice: each chunk's exclusive prefix, in chunk order
            __threadfence();
            const float *src = p.part + (size_t)slice * p.chunks * pst;
            float *pr = p.pre + (size_t)slice * p.chunks * pre_stride(m, d);
            for (int i = threadIdx.x; i < (int)pst; i += blockDim.x) {
                float s = 0.f;
                for (int cc = 0; cc < p.chunks; ++cc) {
                    // pre layout: W [m d] then Delta [m]; part layout: Delta [m] then W [m d]
                    const size_t at = i < m ? md + i : (size_t)(i - m);
                    pr[(size_t)cc * pre_stride(m, d) + at] = s;
                    s = __fadd_rn(s, __ldcg(src + cc * pst + i));
                }
            }
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) atomicExch(p.ready + slice, 1u);
        } else {
            // ------------------------------------------------ C2: the chunk's rows of H
            if (threadIdx.x == 0) {
                const volatile unsigned *flag = p.ready + slice;
                int ok = 1;
                if (*flag == 0u) {
                    const uint64_t t0 = globaltimer_now();
                    while (*flag == 0u) {
                        if (globaltimer_now() - t0 > p.wait_ns) {
                            atomicOr(&g_causal_error, 2u);
                            ok = 0;
                            break;
                        }
                        __nanosleep(256);
                    }
                }
                __threadfence();
                s_flag = ok;
            }
            __syncthreads();
            if (!s_flag) {
                cp_async_commit();  // the U copy issued above has landed before the buffer is reused
                cp_async_wait<0>();
                continue;
            }
            const float *pr = p.pre + ((size_t)slice * p.chunks + c) * pre_stride(m, d);
            for (int i = threadIdx.x * 4; i < (int)md; i += blockDim.x * 4) cp_async16(W + i, pr + i);
            for (int i = threadIdx.x; i < m; i += blockDim.x) Dl[i] = __ldcg(pr + md + i);
            for (int t0 = t_begin; t0 < t_end; t0 += TR) {
                const int rows = min(TR, t_end - t0);
                __syncthreads();
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Vs, V + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                // B[r][l] = A[r][l] / (Delta_l + sum_{r'<=r} A[r'][l]), one thread per anchor
                for (int l = threadIdx.x; l < m; l += blockDim.x) {
                    float run = Dl[l];
                    for (int r = 0; r < rows; ++r) {
                        const float a = As[(size_t)r * ap + l];
                        run = __fadd_rn(run, a);
                        Bs[(size_t)r * ap + l] = run != 0.f ? __fdiv_rn(a, run) : 0.f;
                    }
                }
                __syncthreads();
                // Ht = B W (l ascending); C[r][j] = sum_l B[r][l] A[j][l] for j <= r, else 0
                {
                    const int nct = d / 4, nrt = (rows + 1) / 2;
                    for (int t = threadIdx.x; t < nrt * nct; t += blockDim.x) {
                        const int rt = t / nct, ct = t - rt * nct;
                        const int r0 = rt * 2, k0 = ct * 4, r1 = r0 + 1 < rows ? r0 + 1 : r0;
                        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                        for (int l = 0; l < m; ++l) {
                            const float x0 = Bs[(size_t)r0 * ap + l], x1 = Bs[(size_t)r1 * ap + l];
                            const float4 w = *reinterpret_cast<const float4 *>(W + (size_t)l * d + k0);
                            a.x = __fmaf_rn(x0, w.x, a.x);
                            a.y = __fmaf_rn(x0, w.y, a.y);
                            a.z = __fmaf_rn(x0, w.z, a.z);
                            a.w = __fmaf_rn(x0, w.w, a.w);
                            b.x = __fmaf_rn(x1, w.x, b.x);
                            b.y = __fmaf_rn(x1, w.y, b.y);
                            b.z = __fmaf_rn(x1, w.z, b.z);
                            b.w = __fmaf_rn(x1, w.w, b.w);
                        }
                        *reinterpret_cast<float4 *>(Ht + (size_t)r0 * d + k0) = a;
                        if (r0 + 1 < rows) *reinterpret_cast<float4 *>(Ht + (size_t)(r0 + 1) * d + k0) = b;
                    }
                    for (int t = threadIdx.x; t < rows * rows; t += blockDim.x) {
                        const int r = t / rows, j = t - r * rows;
                        float s = 0.f;
                        if (j <= r)
                            for (int l = 0; l < m; ++l) s = __fmaf_rn(Bs[(size_t)r * ap + l], As[(size_t)j * ap + l], s);
                        Cs[(size_t)r * cp + j] = s;
                    }
                }
                __syncthreads();
                // Ht += C V_tile (j ascending, j <= r), then the rows go out
                {
                    const int nct = d / 8;
                    for (int t = threadIdx.x; t < rows * nct; t += blockDim.x) {
                        const int r = t / nct, k0 = (t - r * nct) * 8;
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = Ht[(size_t)r * d + k0 + e];
                        for (int j = 0; j <= r; ++j) {
                            const float cj = Cs[(size_t)r * cp + j];
                            float y[8];
                            ld8(Vs + (size_t)j * pitch + k0, y);
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = __fmaf_rn(cj, y[e], v[e]);
                        }
                        st8(H + off + (size_t)(t0 + r) * d + k0, v);
                    }
                }
                __syncthreads();
                // the tile joins the prefix
                accumulate(As, ap, Vs, pitch, W, Dl, rows, m, d);
            }
        }
    }
}

template <typename T>
cudaError_t causal_launch_t(const Problem &pr, void *ws, cudaStream_t stream) {
    const int tile = causal_tile<T>(pr.m, pr.d);
    if (tile == 0) return cudaErrorInvalidValue;
    const size_t smem = causal_smem<T>(pr.m, pr.d, tile);
    auto kern = causal_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return e;
    const CausalLayout L = causal_layout(pr);
    CausalParams p;
    p.heads = pr.heads;
    p.n = pr.n;
    p.m = pr.m;
    p.d = pr.d;
    p.scale = pr.scale;
    p.slices = (int)pr.slices();
    p.chunks = (pr.n + kSimtChunk - 1) / kSimtChunk;
    p.tile = tile;
    p.wait_ns = kWaitNs;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.ticket = reinterpret_cast<unsigned *>(w);
    p.arrived = p.ticket + 32;
    p.ready = p.arrived + p.slices;
    p.part = reinterpret_cast<float *>(w + L.part_offset);
    p.pre = reinterpret_cast<float *>(w + L.pre_offset);
    const long long items = 2LL * p.slices * p.chunks;
    const int grid = (int)std::min<long long>((long long)sms * std::max(per_sm, 1), items);
    if ((e = cudaMemsetAsync(ws, 0, L.header_bytes, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>((const T *)pr.Q, (const T *)pr.U, (const T *)pr.V, (T *)pr.H, p);
    return cudaGetLastError();
}

}  // namespace

bool causal_fits(const Problem &p) {
    return (p.f32 ? causal_tile<float>(p.m, p.d) : causal_tile<__nv_bfloat16>(p.m, p.d)) > 0;
}

CausalLayout causal_layout(const Problem &p) {
    CausalLayout L;
    const size_t S = (size_t)p.slices();
    const size_t chunks = (p.n + kSimtChunk - 1) / kSimtChunk;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    L.header_bytes = up((32 + 2 * S) * 4);
    L.part_offset = L.header_bytes;
    L.pre_offset = up(L.part_offset + 4 * S * chunks * ((size_t)p.m + (size_t)p.m * p.d));
    L.total_bytes = L.pre_offset + 4 * S * chunks * pre_stride(p.m, p.d);
    return L;
}

cudaError_t launch_causal(const Problem &p, void *workspace, cudaStream_t stream) {
    return p.f32 ? causal_launch_t<float>(p, workspace, stream) : causal_launch_t<__nv_bfloat16>(p, workspace, stream);
}

cudaError_t causal_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_causal_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_causal_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

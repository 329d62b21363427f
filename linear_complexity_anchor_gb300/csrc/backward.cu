// Backward of the anchor-attention forward on CUDA cores (fp32 FMA): for an upstream gradient
// dH of H = A Delta^{-1} (A^T V), A = rowsoftmax(scale Q U^T), the gradients
//   dW' = A^T dH,  dW = Delta^{-1} dW',  dDelta_j = -sum_k dW'[j][k] W'[j][k] / Delta_j,
//   G = dH W'^T + V dW^T + 1 dDelta^T,  dS = A o (G - rowsum(A o G)),
//   dQ = scale dS U,  dV = A dW,  dU = scale dS^T Q summed over the batch entries of a head.
// (The anchors are fitted by gradient descent: pith.science verdict on arXiv 2505.16463,
// "core_discovery"; the arXiv abstract, where the anchors are weights of a trainable layer.)
//
// Two launches:
//   anchor_bwd_kernel    work items from a ticket, in a fixed order: every B1 item (a
//                        512-token chunk of a slice: A recomputed, and its partial Delta,
//                        A^T V and A^T dH), then every B2 item (the same 512 tokens: A
//                        recomputed, G, dS, the chunk's dQ and dV rows, and its dU partial).
//                        The last B1 chunk of a slice to finish sums the slice's partials in
//                        chunk order and publishes W', dW and dDelta; a B2 item waits for them
//                        (bounded).  A B2 item only waits for B1 items held by running CTAs.
//   anchor_bwd_du_kernel dU of each head: the B2 partials of its slices summed in a fixed
//                        (batch, chunk) order.
// Every contraction keeps one accumulator per output and adds its terms in ascending index
// order, so results are bit-identical from run to run.
#include "common.cuh"
#include "simt_ops.cuh"

#include <math.h>

namespace anchor {

// Device error word of the backward (bit 1: a wait for a slice's reduction gave up).
__device__ unsigned int g_bwd_error;

namespace {

using namespace simt;

constexpr int kThreads = 256;
constexpr int kDuSlots = 8;  // dU outputs per thread are kept in registers: m d <= 16384 = 256 x 8 x 8
constexpr uint64_t kWaitNs = 2000000000ull;

// floats per slice of the published W' | dW | dDelta block: read with 16-byte copies
__host__ __device__ __forceinline__ size_t pub_stride(int m, int d) { return 2 * (size_t)m * d + ((m + 3) & ~3); }

struct BwdParams {
    int heads, n, m, d;
    float scale;
    int slices, chunks, tile;
    unsigned *ticket;    // next work item
    unsigned *arrived;   // [slices] B1 chunks finished
    unsigned *ready;     // [slices] W', dW, dDelta published
    float *part;         // [slices][chunks][m + 2 m d]  Delta | A^T V | A^T dH
    float *pub;          // [slices][2 m d + m4]         W' | dW | dDelta (m4: m rounded up to 4)
    float *dupart;       // [slices][chunks][m d]        scale dS^T Q of a chunk
    uint64_t wait_ns;
};

// G[r][j] = dDelta_j + sum_k (dH[r][k] W'[j][k] + V[r][k] dW[j][k]) (k ascending) into Gs,
// r < rows, j < m.  Tiles of 4 rows x 4 anchors as in the scores.
template <typename T>
__device__ __forceinline__ void grad_a(const T *dHs, const T *Vs, int pitch, const float *Wp, const float *dW,
                                       const float *dD, float *Gs, int ap, int rows, int m, int d) {
    const int nct = (m + 3) / 4, nrt = (rows + 3) / 4;
    for (int t = threadIdx.x; t < nrt * nct; t += blockDim.x) {
        const int rt = t / nct, ct = t - rt * nct;
        const T *h[4], *v[4];
        const float *w[4], *g[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = min(rt + i * nrt, rows - 1), j = min(ct + i * nct, m - 1);
            h[i] = dHs + (size_t)r * pitch;
            v[i] = Vs + (size_t)r * pitch;
            w[i] = Wp + (size_t)j * d;
            g[i] = dW + (size_t)j * d;
        }
        float acc[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float base = dD[min(ct + b * nct, m - 1)];
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a][b] = base;
        }
        for (int k = 0; k < d; k += 4) {
            float4 ha[4], va[4], wa[4], ga[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ha[i] = ld4(h[i] + k);
                va[i] = ld4(v[i] + k);
                wa[i] = ld4(w[i] + k);
                ga[i] = ld4(g[i] + k);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float s = acc[a][b];
                    s = __fmaf_rn(ha[a].x, wa[b].x, s);
                    s = __fmaf_rn(va[a].x, ga[b].x, s);
                    s = __fmaf_rn(ha[a].y, wa[b].y, s);
                    s = __fmaf_rn(va[a].y, ga[b].y, s);
                    s = __fmaf_rn(ha[a].z, wa[b].z, s);
                    s = __fmaf_rn(va[a].z, ga[b].z, s);
                    s = __fmaf_rn(ha[a].w, wa[b].w, s);
                    acc[a][b] = __fmaf_rn(va[a].w, ga[b].w, s);
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int r = rt + a * nrt, j = ct + b * nct;
                if (r < rows && j < m) Gs[(size_t)r * ap + j] = acc[a][b];
            }
    }
}

// dS = A o (G - sum_l A_l G_l) in place of G, one thread per row (l ascending)
__device__ __forceinline__ void softmax_grad(const float *As, float *Gs, int ap, int rows, int m) {
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        const float *a = As + (size_t)r * ap;
        float *g = Gs + (size_t)r * ap;
        float s = 0.f;
        for (int j = 0; j < m; ++j) s = __fmaf_rn(a[j], g[j], s);
        for (int j = 0; j < m; ++j) g[j] = __fmul_rn(a[j], __fsub_rn(g[j], s));
    }
}

// acc[slot] += sum_r dS[r][j] Q[r][k] for this thread's (2 anchors x 4 columns) tiles
// t = threadIdx.x + slot * blockDim.x (r ascending)
template <typename T>
__device__ __forceinline__ void accumulate_du(const float *Ds, int ap, const T *Qs, int pitch, float (&acc)[kDuSlots][8],
                                              int rows, int m, int d) {
    const int nct = d / 4, njt = (m + 1) / 2;
#pragma unroll
    for (int sl = 0; sl < kDuSlots; ++sl) {
        const int t = threadIdx.x + sl * blockDim.x;
        if (t >= njt * nct) break;
        const int jt = t / nct, ct = t - jt * nct;
        const int j0 = jt * 2, k0 = ct * 4, j1 = j0 + 1 < m ? j0 + 1 : j0;
        for (int r = 0; r < rows; ++r) {
            const float a0 = Ds[(size_t)r * ap + j0], a1 = Ds[(size_t)r * ap + j1];
            const float4 q = ld4(Qs + (size_t)r * pitch + k0);
            acc[sl][0] = __fmaf_rn(a0, q.x, acc[sl][0]);
            acc[sl][1] = __fmaf_rn(a0, q.y, acc[sl][1]);
            acc[sl][2] = __fmaf_rn(a0, q.z, acc[sl][2]);
            acc[sl][3] = __fmaf_rn(a0, q.w, acc[sl][3]);
            acc[sl][4] = __fmaf_rn(a1, q.x, acc[sl][4]);
            acc[sl][5] = __fmaf_rn(a1, q.y, acc[sl][5]);
            acc[sl][6] = __fmaf_rn(a1, q.z, acc[sl][6]);
            acc[sl][7] = __fmaf_rn(a1, q.w, acc[sl][7]);
        }
    }
}

// Shared memory: U [m][pitch] (input type) | M1 [m][d] | M2 [m][d] | Dm [m, padded to 4] (fp32) |
// Q, V, dH tiles [TR][pitch] (input type) | A [TR][m+1] | G [TR][m+1] (fp32).  B1: M1 = A^T V,
// M2 = A^T dH, Dm = Delta; B2: M1 = W', M2 = dW, Dm = dDelta.
template <typename T> size_t bwd_smem(int m, int d, int tile) {
    const size_t pitch = d + pad_elems<T>();
    return sizeof(T) * ((size_t)m + 3 * tile) * pitch +
           4 * (2 * (size_t)m * d + ((m + 3) & ~3) + 2 * (size_t)tile * (m + 1));
}

template <typename T> int bwd_tile(int m, int d) {
    for (int tile = 64; tile >= 4; tile /= 2)
        if (bwd_smem<T>(m, d, tile) <= kSimtMaxSmem) return tile;
    return 0;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
anchor_bwd_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V, const T *__restrict__ dH,
                  T *__restrict__ dQ, T *__restrict__ dV, const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ unsigned s_item;
    __shared__ int s_flag;
    const int m = p.m, d = p.d, TR = p.tile;
    const int pitch = d + pad_elems<T>();
    const int ap = m + 1;
    T *Us = reinterpret_cast<T *>(smem);
    float *M1 = reinterpret_cast<float *>(Us + (size_t)m * pitch);
    float *M2 = M1 + (size_t)m * d;
    float *Dm = M2 + (size_t)m * d;
    T *Qs = reinterpret_cast<T *>(Dm + ((m + 3) & ~3));
    T *Vs = Qs + (size_t)TR * pitch;
    T *Hs = Vs + (size_t)TR * pitch;
    float *As = reinterpret_cast<float *>(Hs + (size_t)TR * pitch);
    float *Gs = As + (size_t)TR * ap;
    const unsigned n1 = (unsigned)(p.slices * p.chunks);
    const size_t pstride = (size_t)m + 2 * (size_t)m * d;
    const size_t md = (size_t)m * d;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_item = atomicAdd(p.ticket, 1u);
        __syncthreads();
        const unsigned item = s_item;
        if (item >= 2 * n1) break;
        const bool b1 = item < n1;
        const unsigned it = b1 ? item : item - n1;
        const int slice = (int)(it / p.chunks), c = (int)(it % p.chunks);
        const int h = slice % p.heads;
        const size_t off = (size_t)slice * p.n * d;
        const int t_begin = c * kSimtChunk, t_end = min(p.n, t_begin + kSimtChunk);
        if (b1) {
            // ------------------------------------------------ B1: Delta, A^T V, A^T dH partials
            stage_rows(Us, U + (size_t)h * md, m, d, pitch);
            cp_async_commit();
            for (int i = threadIdx.x; i < (int)(2 * md) + m; i += blockDim.x) M1[i] = 0.f;  // M1, M2, Dm
            for (int t0 = t_begin; t0 < t_end; t0 += TR) {
                const int rows = min(TR, t_end - t0);
                __syncthreads();
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Vs, V + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Hs, dH + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                accumulate(As, ap, Vs, pitch, M1, Dm, rows, m, d);
                accumulate(As, ap, Hs, pitch, M2, static_cast<float *>(nullptr), rows, m, d);
            }
            __syncthreads();
            float *dst = p.part + ((size_t)slice * p.chunks + c) * pstride;
            for (int i = threadIdx.x; i < m; i += blockDim.x) dst[i] = Dm[i];
            for (int i = threadIdx.x; i < (int)(2 * md); i += blockDim.x) dst[m + i] = M1[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_flag = atomicAdd(p.arrived + slice, 1u) == (unsigned)(p.chunks - 1);
            __syncthreads();
            if (!s_flag) continue;
            // last chunk of the slice: sums in chunk order, then W', dW and dDelta
            __threadfence();
            const float *src = p.part + (size_t)slice * p.chunks * pstride;
            for (int i = threadIdx.x; i < (int)pstride; i += blockDim.x) {
                float s = 0.f;
                for (int cc = 0; cc < p.chunks; ++cc) s = __fadd_rn(s, __ldcg(src + cc * pstride + i));
                if (i < m) Dm[i] = s;
                else M1[i - m] = s;  // M1 then M2, contiguous
            }
            __syncthreads();
            // W' = W / Delta, dW = dW' / Delta (0 where Delta = 0)
            for (int i = threadIdx.x; i < (int)md; i += blockDim.x) {
                const float dj = Dm[i / d];
                M1[i] = dj != 0.f ? __fdiv_rn(M1[i], dj) : 0.f;
                M2[i] = dj != 0.f ? __fdiv_rn(M2[i], dj) : 0.f;
            }
            __syncthreads();
            // dDelta_j = -sum_k dW'_jk W'_jk / Delta_j = -sum_k dW_jk W'_jk (k ascending)
            for (int j = threadIdx.x; j < m; j += blockDim.x) {
                float s = 0.f;
                for (int k = 0; k < d; ++k) s = __fmaf_rn(M2[(size_t)j * d + k], M1[(size_t)j * d + k], s);
                Dm[j] = Dm[j] != 0.f ? -s : 0.f;
            }
            __syncthreads();
            float *pb = p.pub + (size_t)slice * pub_stride(m, d);
            for (int i = threadIdx.x; i < (int)(2 * md) + m; i += blockDim.x) pb[i] = M1[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) atomicExch(p.ready + slice, 1u);
        } else {
            // ------------------------------------------------ B2: dQ, dV rows and a dU partial
            if (threadIdx.x == 0) {
                // every B1 item was handed out before this one, to CTAs that are running
                const volatile unsigned *flag = p.ready + slice;
                int ok = 1;
                if (*flag == 0u) {
                    const uint64_t t0 = globaltimer_now();
                    while (*flag == 0u) {
                        if (globaltimer_now() - t0 > p.wait_ns) {
                            atomicOr(&g_bwd_error, 2u);
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
            if (!s_flag) continue;  // this chunk's dQ, dV and dU share stay unwritten; the error word says why
            stage_rows(Us, U + (size_t)h * md, m, d, pitch);
            const float *pb = p.pub + (size_t)slice * pub_stride(m, d);  // a multiple of 16 bytes
            for (int i = threadIdx.x * 4; i < (int)(2 * md); i += blockDim.x * 4) cp_async16(M1 + i, pb + i);
            for (int i = threadIdx.x; i < m; i += blockDim.x) Dm[i] = __ldcg(pb + 2 * md + i);
            float acc[kDuSlots][8];
#pragma unroll
            for (int sl = 0; sl < kDuSlots; ++sl)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[sl][e] = 0.f;
            for (int t0 = t_begin; t0 < t_end; t0 += TR) {
                const int rows = min(TR, t_end - t0);
                __syncthreads();
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Vs, V + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Hs, dH + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                grad_a(Hs, Vs, pitch, M1, M2, Dm, Gs, ap, rows, m, d);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                softmax_grad(As, Gs, ap, rows, m);
                __syncthreads();
                apply(Gs, ap, Us, pitch, dQ + off + (size_t)t0 * d, rows, m, d, p.scale);  // dQ = scale dS U
                apply(As, ap, M2, d, dV + off + (size_t)t0 * d, rows, m, d, 1.f);           // dV = A dW
                accumulate_du(Gs, ap, Qs, pitch, acc, rows, m, d);
            }
            // this chunk's share of dU (scale dS^T Q): written whole, summed by the second launch
            float *du = p.dupart + ((size_t)slice * p.chunks + c) * md;
            const int nct = d / 4, njt = (m + 1) / 2;
#pragma unroll
            for (int sl = 0; sl < kDuSlots; ++sl) {
                const int t = threadIdx.x + sl * blockDim.x;
                if (t >= njt * nct) break;
                const int jt = t / nct, ct = t - jt * nct;
                const int j0 = jt * 2, k0 = ct * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) du[(size_t)j0 * d + k0 + e] = __fmul_rn(p.scale, acc[sl][e]);
                if (j0 + 1 < m)
#pragma unroll
                    for (int e = 0; e < 4; ++e) du[(size_t)(j0 + 1) * d + k0 + e] = __fmul_rn(p.scale, acc[sl][4 + e]);
            }
        }
    }
}

// dU[h][e] = sum over the K = B chunks shares k = (b, c) (b-major) of dupart[b heads + h][c][e],
// in a fixed order: a CTA takes 32 consecutive e (one coalesced 128-byte row per share) and 8
// groups of shares; group g adds shares g, g + 8, g + 16, ... in that order (loads issued 8 at
// a time), then group 0 adds the 8 group sums in group order.
constexpr int kDuGroups = 8, kDuBatch = 8;
template <typename T>
__global__ void __launch_bounds__(32 * kDuGroups)
anchor_bwd_du_kernel(const float *__restrict__ dupart, T *__restrict__ dU, int B, int heads, int chunks, int md) {
    __shared__ float part[kDuGroups][32];
    // launched with programmatic stream serialization after the kernel that writes dupart
    grid_dependency_wait();
    grid_dependents_launch();
    const int h = blockIdx.y, lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const int K = B * chunks;
    float s = 0.f;
    if (e < md) {
        for (int k0 = g; k0 < K; k0 += kDuGroups * kDuBatch) {
            float x[kDuBatch];
#pragma unroll
            for (int u = 0; u < kDuBatch; ++u) {
                const int k = k0 + u * kDuGroups;
                const int b = k / chunks, c = k - b * chunks;
                x[u] = k < K ? __ldg(dupart + ((size_t)(b * heads + h) * chunks + c) * md + e) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kDuBatch; ++u)
                if (k0 + u * kDuGroups < K) s = __fadd_rn(s, x[u]);
        }
    }
    part[g][lane] = s;
    __syncthreads();
    if (g == 0 && e < md) {
        float t = part[0][lane];
#pragma unroll
        for (int q = 1; q < kDuGroups; ++q) t = __fadd_rn(t, part[q][lane]);
        dU[(size_t)h * md + e] = from_f32<T>(t);
    }
}

template <typename T>
cudaError_t bwd_launch(const BwdProblem &p, void *ws, cudaStream_t stream) {
    const int tile = bwd_tile<T>(p.m, p.d);
    if (tile == 0) return cudaErrorInvalidValue;
    const size_t smem = bwd_smem<T>(p.m, p.d, tile);
    auto kern = anchor_bwd_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return e;
    const BwdLayout L = bwd_layout(p);
    BwdParams bp;
    bp.heads = p.heads;
    bp.n = p.n;
    bp.m = p.m;
    bp.d = p.d;
    bp.scale = p.scale;
    bp.slices = (int)p.slices();
    bp.chunks = (p.n + kSimtChunk - 1) / kSimtChunk;
    bp.tile = tile;
    bp.wait_ns = kWaitNs;
    uint8_t *w = static_cast<uint8_t *>(ws);
    bp.ticket = reinterpret_cast<unsigned *>(w);
    bp.arrived = bp.ticket + 32;
    bp.ready = bp.arrived + bp.slices;
    bp.part = reinterpret_cast<float *>(w + L.part_offset);
    bp.pub = reinterpret_cast<float *>(w + L.pub_offset);
    bp.dupart = reinterpret_cast<float *>(w + L.dupart_offset);
    const long long items = 2LL * bp.slices * bp.chunks;
    const int grid = (int)std::min<long long>((long long)sms * std::max(per_sm, 1), items);
    if ((e = cudaMemsetAsync(ws, 0, L.header_bytes, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>((const T *)p.Q, (const T *)p.U, (const T *)p.V, (const T *)p.dH, (T *)p.dQ,
                                           (T *)p.dV, bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_bwd_du_sum(bp.dupart, p.dU, p.B, p.heads, bp.chunks, p.m * p.d, p.f32, stream);
}

}  // namespace

bool bwd_fits(const BwdProblem &p) {
    return (p.f32 ? bwd_tile<float>(p.m, p.d) : bwd_tile<__nv_bfloat16>(p.m, p.d)) > 0;
}

BwdLayout bwd_layout(const BwdProblem &p) {
    BwdLayout L;
    const size_t S = (size_t)p.slices();
    const size_t chunks = (p.n + kSimtChunk - 1) / kSimtChunk;
    const size_t md = (size_t)p.m * p.d;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    L.header_bytes = up((32 + 2 * S) * 4);
    L.part_offset = L.header_bytes;
    L.pub_offset = up(L.part_offset + 4 * S * chunks * (p.m + 2 * md));
    L.dupart_offset = up(L.pub_offset + 4 * S * pub_stride(p.m, p.d));
    L.total_bytes = L.dupart_offset + 4 * S * chunks * md;
    return L;
}

cudaError_t launch_bwd(const BwdProblem &p, void *workspace, cudaStream_t stream) {
    return p.f32 ? bwd_launch<float>(p, workspace, stream) : bwd_launch<__nv_bfloat16>(p, workspace, stream);
}

cudaError_t launch_bwd_du_sum(const float *dupart, void *dU, int B, int heads, int chunks, int md, bool f32,
                              cudaStream_t stream) {
    const dim3 grid((md + 31) / 32, heads);
    if (f32)
        return launch_pdl(anchor_bwd_du_kernel<float>, grid, dim3(32 * kDuGroups), 0, stream, dupart, (float *)dU, B,
                          heads, chunks, md);
    return launch_pdl(anchor_bwd_du_kernel<__nv_bfloat16>, grid, dim3(32 * kDuGroups), 0, stream, dupart,
                      (__nv_bfloat16 *)dU, B, heads, chunks, md);
}

cudaError_t bwd_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

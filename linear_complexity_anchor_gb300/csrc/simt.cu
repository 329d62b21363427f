// CUDA-core (fp32 FMA) variants of the anchor-attention forward
//   H = A Delta^{-1} (A^T V),  A = rowsoftmax(scale * Q U^T),  Delta = diag(colsum A)
// (AnchorFormer, arXiv 2505.16463; pith.science verdict, "key_machinery" and the referee
// summary of Eq. 11/12).  Used for the fp32 entry point, for m < 32 (where a tensor-core
// tile would be mostly padding), for d in {16, 32} and for a non-positive scale.
//
// Two kernels, both one launch per call:
//   simt_full_kernel   one CTA per (batch, head) slice with the whole slice in shared memory:
//                      Q, V and U arrive by cp.async (16-byte copies), and every step runs
//                      on chip (scores, softmax, Delta, A^T V, Delta^{-1}, A W').  No workspace.
//   simt_chunk_kernel  slices too long for shared memory.  Work items are handed out by a
//                      ticket in a fixed order: every P1 item (a 512-token chunk of a slice:
//                      its partial Delta and A^T V), then every P2 item (64 tokens of a slice:
//                      A recomputed with the same code, H = A W').  The last P1 chunk of a
//                      slice to finish sums the slice's partials in chunk order and publishes
//                      W' = Delta^{-1} A^T V; a P2 item waits for it (bounded).  A P2 item only
//                      waits for P1 items that running CTAs already hold, so no grid size can
//                      deadlock, and the sums do not depend on which CTA ran what.
// Every contraction keeps one accumulator per output and adds its terms in ascending index
// order (register tiles of outputs, 16-byte shared-memory operand loads), so results are
// bit-identical from run to run.
#include "common.cuh"
#include "simt_ops.cuh"

#include <math.h>

namespace anchor {

// Device error word of the chunked kernel (bit 1: a wait for a slice's W' gave up).
__device__ unsigned int g_simt_error;

namespace {

using namespace simt;

constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // a wait for another CTA's reduction gives up after 2 s

// ------------------------------------------------------------------ whole slice per CTA
// Shared memory of a whole slice: Qs | Vs | Us | Ws | Ds | As, or (kOver) with As laid over Qs
// (the scores are formed in registers first), small enough for three CTAs per SM.
template <typename T, bool kOver>
__device__ __host__ __forceinline__ size_t full_qa_bytes(int n, int m, int d) {
    const size_t q = sizeof(T) * (size_t)n * (d + pad_elems<T>()), a = 4 * (size_t)n * (m + 1);
    return kOver ? ((q > a ? q : a) + 15) / 16 * 16 : q;
}

template <typename T, bool kOver>
__global__ void __launch_bounds__(kThreads, kOver ? 3 : 2)
simt_full_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V, T *__restrict__ H,
                 int heads, int n, int m, int d, float scale) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int pitch = d + pad_elems<T>();
    const int ap = m + 1;
    T *Qs = reinterpret_cast<T *>(smem);                    // [n][pitch]
    T *Vs = reinterpret_cast<T *>(smem + full_qa_bytes<T, kOver>(n, m, d));  // [n][pitch]
    T *Us = Vs + (size_t)n * pitch;                         // [m][pitch]
    float *Ws = reinterpret_cast<float *>(Us + (size_t)m * pitch);  // [m][d]  A^T V, then W'
    float *Ds = Ws + (size_t)m * d;                         // [m]     Delta
    float *As = kOver ? reinterpret_cast<float *>(smem) : Ds + ((m + 3) & ~3);  // [n][ap]
    const long long slice = blockIdx.x;
    const int h = (int)(slice % heads);
    const size_t off = (size_t)slice * n * d;

    // launched with programmatic stream serialization: global memory only from here on
    grid_dependency_wait();
    grid_dependents_launch();
    stage_rows(Qs, Q + off, n, d, pitch);
    stage_rows(Us, U + (size_t)h * m * d, m, d, pitch);
    cp_async_commit();
    stage_rows(Vs, V + off, n, d, pitch);  // lands while the scores are computed
    cp_async_commit();
    for (int p = threadIdx.x; p < m * d + m; p += blockDim.x) Ws[p] = 0.f;  // and Ds
    cp_async_wait<1>();
    __syncthreads();
    if (kOver) scores_over(Qs, Us, pitch, As, ap, n, m, d, scale);
    else scores(Qs, Us, pitch, As, ap, n, m, d, scale);
    __syncthreads();
    softmax_rows(As, ap, n, m);
    cp_async_wait<0>();
    __syncthreads();
    accumulate(As, ap, Vs, pitch, Ws, Ds, n, m, d);
    __syncthreads();
    normalise(Ws, Ds, m, d);
    __syncthreads();
    apply(As, ap, Ws, d, H + off, n, m, d, 1.f);
}

// ------------------------------------------------------------------ chunked slices
struct ChunkParams {
    int heads, n, m, d;
    float scale;
    int slices, chunks, blocks;  // P1 chunks and P2 blocks per slice
    int tile;                    // tokens per staged tile (64 unless the anchors need the room)
    unsigned *ticket;            // next work item
    unsigned *arrived;           // [slices] P1 chunks finished
    unsigned *ready;             // [slices] W' published
    float *part;                 // [slices][chunks][m * d + m]  A^T V and Delta partials
    float *wprime;               // [slices][m * d]
    uint64_t wait_ns;
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
simt_chunk_kernel(const T *__restrict__ Q, const T *__restrict__ U, const T *__restrict__ V, T *__restrict__ H,
                  const ChunkParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ unsigned s_item;
    __shared__ int s_flag;
    const int m = p.m, d = p.d, TR = p.tile;
    const int pitch = d + pad_elems<T>();
    const int ap = m + 1;
    T *Us = reinterpret_cast<T *>(smem);                    // [m][pitch]
    T *Qs = Us + (size_t)m * pitch;                         // [TR][pitch]
    T *Vs = Qs + (size_t)TR * pitch;                        // [TR][pitch]
    float *Wacc = reinterpret_cast<float *>(Vs + (size_t)TR * pitch);  // [m][d]  partial / W'
    float *Dacc = Wacc + (size_t)m * d;                     // [m]
    float *As = Dacc + ((m + 3) & ~3);                      // [TR][ap]
    const unsigned n1 = (unsigned)(p.slices * p.chunks), n2 = (unsigned)(p.slices * p.blocks);
    const size_t pstride = (size_t)m * d + m;

    for (;;) {
        __syncthreads();  // the previous item is done with shared memory and s_item
        if (threadIdx.x == 0) s_item = atomicAdd(p.ticket, 1u);
        __syncthreads();
        const unsigned item = s_item;
        if (item >= n1 + n2) break;
        if (item < n1) {
            // ---------------------------------------------------------- P1: a chunk's partial
            const int slice = (int)(item / p.chunks), c = (int)(item % p.chunks);
            const int h = slice % p.heads;
            const size_t off = (size_t)slice * p.n * d;
            const int t_begin = c * kSimtChunk, t_end = min(p.n, t_begin + kSimtChunk);
            stage_rows(Us, U + (size_t)h * m * d, m, d, pitch);
            cp_async_commit();
            for (int i = threadIdx.x; i < m * d + m; i += blockDim.x) Wacc[i] = 0.f;  // and Dacc
            for (int t0 = t_begin; t0 < t_end; t0 += TR) {
                const int rows = min(TR, t_end - t0);
                __syncthreads();  // the last tile's Vs and As are read
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                stage_rows(Vs, V + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                accumulate(As, ap, Vs, pitch, Wacc, Dacc, rows, m, d);
            }
            __syncthreads();
            float *dst = p.part + ((size_t)slice * p.chunks + c) * pstride;
            for (int i = threadIdx.x; i < m * d + m; i += blockDim.x) dst[i] = Wacc[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_flag = atomicAdd(p.arrived + slice, 1u) == (unsigned)(p.chunks - 1);
            __syncthreads();
            if (!s_flag) continue;
            // the last chunk of the slice: sum every partial in chunk order, then publish W'
            __threadfence();
            const float *src = p.part + (size_t)slice * p.chunks * pstride;
            for (int i = threadIdx.x; i < m * d + m; i += blockDim.x) {
                float s = 0.f;
                for (int cc = 0; cc < p.chunks; ++cc) s = __fadd_rn(s, __ldcg(src + cc * pstride + i));
                Wacc[i] = s;
            }
            __syncthreads();
            normalise(Wacc, Dacc, m, d);
            __syncthreads();
            float *wp = p.wprime + (size_t)slice * m * d;
            for (int i = threadIdx.x; i < m * d; i += blockDim.x) wp[i] = Wacc[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) atomicExch(p.ready + slice, 1u);
        } else {
            // ---------------------------------------------------------- P2: 64 tokens of H
            const unsigned it2 = item - n1;
            const int slice = (int)(it2 / p.blocks), blk = (int)(it2 % p.blocks);
            const int h = slice % p.heads;
            const size_t off = (size_t)slice * p.n * d;
            if (threadIdx.x == 0) {
                // every P1 item was handed out before this one, to CTAs that are running
                const volatile unsigned *flag = p.ready + slice;
                int ok = 1;
                if (*flag == 0u) {
                    const uint64_t t0 = globaltimer_now();
                    while (*flag == 0u) {
                        if (globaltimer_now() - t0 > p.wait_ns) {
                            atomicOr(&g_simt_error, 2u);
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
            if (!s_flag) continue;  // H of this block stays unwritten; the error word says why
            stage_rows(Us, U + (size_t)h * m * d, m, d, pitch);
            const float *wp = p.wprime + (size_t)slice * m * d;
            for (int i = threadIdx.x * 4; i < m * d; i += blockDim.x * 4)
                cp_async16(Wacc + i, wp + i);
            for (int t0 = blk * 64; t0 < min(p.n, blk * 64 + 64); t0 += TR) {
                const int rows = min(TR, p.n - t0);
                __syncthreads();
                stage_rows(Qs, Q + off + (size_t)t0 * d, rows, d, pitch);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                scores(Qs, Us, pitch, As, ap, rows, m, d, p.scale);
                __syncthreads();
                softmax_rows(As, ap, rows, m);
                __syncthreads();
                apply(As, ap, Wacc, d, H + off + (size_t)t0 * d, rows, m, d, 1.f);
            }
        }
    }
}

template <typename T, bool kOver = false> size_t full_smem(int n, int m, int d) {
    const size_t pitch = d + pad_elems<T>();
    return full_qa_bytes<T, kOver>(n, m, d) + sizeof(T) * ((size_t)n + m) * pitch +
           4 * ((size_t)m * d + ((m + 3) & ~3) + (kOver ? 0 : (size_t)n * (m + 1)));
}
// the compact layout when it fits three CTAs per SM and the scores' tiles two per thread
template <typename T> bool full_over(int n, int m, int d) {
    return full_smem<T, true>(n, m, d) <= kSimtThirdSmem &&
           (long long)((n + 3) / 4) * ((m + 3) / 4) <= 2LL * kThreads;
}

template <typename T> size_t chunk_smem(int m, int d, int tile) {
    const size_t pitch = d + pad_elems<T>();
    return sizeof(T) * ((size_t)m + 2 * tile) * pitch + 4 * ((size_t)m * d + ((m + 3) & ~3) + (size_t)tile * (m + 1));
}

template <typename T> int chunk_tile(int m, int d) {
    for (int tile = 64; tile >= 8; tile /= 2)
        if (chunk_smem<T>(m, d, tile) <= kSimtMaxSmem) return tile;
    return 0;
}

template <typename T, bool kOver>
cudaError_t full_launch_t(const Problem &p, cudaStream_t stream) {
    const size_t smem = full_smem<T, kOver>(p.n, p.m, p.d);
    cudaError_t e =
        cudaFuncSetAttribute(simt_full_kernel<T, kOver>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(simt_full_kernel<T, kOver>, dim3((unsigned)p.slices()), dim3(kThreads), smem, stream,
                      (const T *)p.Q, (const T *)p.U, (const T *)p.V, (T *)p.H, p.heads, p.n, p.m, p.d, p.scale);
}
template <typename T>
cudaError_t full_launch(const Problem &p, cudaStream_t stream) {
    return full_over<T>(p.n, p.m, p.d) ? full_launch_t<T, true>(p, stream) : full_launch_t<T, false>(p, stream);
}

template <typename T>
cudaError_t chunk_launch(const Problem &p, void *ws, cudaStream_t stream) {
    const int tile = chunk_tile<T>(p.m, p.d);
    if (tile == 0) return cudaErrorInvalidValue;
    const size_t smem = chunk_smem<T>(p.m, p.d, tile);
    auto kern = simt_chunk_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return e;
    ChunkParams cp;
    cp.heads = p.heads;
    cp.n = p.n;
    cp.m = p.m;
    cp.d = p.d;
    cp.scale = p.scale;
    cp.slices = (int)p.slices();
    cp.chunks = (p.n + kSimtChunk - 1) / kSimtChunk;
    cp.blocks = (p.n + 63) / 64;
    cp.tile = tile;
    cp.wait_ns = kWaitNs;
    const SimtLayout L = simt_chunk_layout(p);
    uint8_t *w = static_cast<uint8_t *>(ws);
    cp.ticket = reinterpret_cast<unsigned *>(w);
    cp.arrived = cp.ticket + 32;
    cp.ready = cp.arrived + cp.slices;
    cp.part = reinterpret_cast<float *>(w + L.part_offset);
    cp.wprime = reinterpret_cast<float *>(w + L.wprime_offset);
    const long long items = (long long)cp.slices * (cp.chunks + cp.blocks);
    const int grid = (int)std::min<long long>((long long)sms * std::max(per_sm, 1), items);
    if ((e = cudaMemsetAsync(ws, 0, L.header_bytes, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>((const T *)p.Q, (const T *)p.U, (const T *)p.V, (T *)p.H, cp);
    return cudaGetLastError();
}

}  // namespace

bool simt_full_fits(const Problem &p) {
    return (p.f32 ? full_smem<float>(p.n, p.m, p.d) : full_smem<__nv_bfloat16>(p.n, p.m, p.d)) <= kSimtMaxSmem;
}

bool simt_chunk_fits(const Problem &p) {
    return (p.f32 ? chunk_tile<float>(p.m, p.d) : chunk_tile<__nv_bfloat16>(p.m, p.d)) > 0;
}

SimtLayout simt_chunk_layout(const Problem &p) {
    SimtLayout L;
    const size_t S = (size_t)p.slices();
    const size_t chunks = (p.n + kSimtChunk - 1) / kSimtChunk;
    L.header_bytes = ((32 + 2 * S) * 4 + 255) / 256 * 256;
    L.part_offset = L.header_bytes;
    // W' is read with 16-byte copies: its region starts on a 256-byte boundary (the partials
    // before it are m d + m floats per chunk, not a multiple of 16 bytes for odd m)
    L.wprime_offset = (L.part_offset + 4 * S * chunks * ((size_t)p.m * p.d + p.m) + 255) / 256 * 256;
    L.total_bytes = L.wprime_offset + 4 * S * (size_t)p.m * p.d;
    return L;
}

cudaError_t launch_simt_full(const Problem &p, cudaStream_t stream) {
    return p.f32 ? full_launch<float>(p, stream) : full_launch<__nv_bfloat16>(p, stream);
}

cudaError_t launch_simt_chunk(const Problem &p, void *workspace, cudaStream_t stream) {
    return p.f32 ? chunk_launch<float>(p, workspace, stream) : chunk_launch<__nv_bfloat16>(p, workspace, stream);
}

cudaError_t simt_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_simt_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_simt_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

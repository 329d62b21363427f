// Anchor-attention forward, one CTA per (batch, head) slice streaming the slice's tiles: the
// tensor-core variant for d = 64, m <= 64 with long slices (bf16 operands, fp32 accumulators
// in tensor memory).  H = A Delta^{-1} (A^T V), A = rowsoftmax(scale Q U^T), evaluated as
// A (Delta^{-1} (A^T V)) (pith.science verdict on arXiv 2505.16463, "key_machinery" and the
// referee summary of Eq. 11/12).
//
// Pass 1 walks the slice's 128-token tiles: S_t = Q_t U^T, A_t = softmax (row warps, bf16),
// [W | Delta] += A_t^T [V_t | 1]; each A_t tile also goes to a workspace by TMA (it stays in
// L2).  Then W' = Delta^{-1} W.  Pass 2 loads the A tiles back and forms H_t = A_t W',
// stored by TMA.  No other CTA takes part in a slice, so nothing waits on another CTA: the
// whole slice's sums run in one tensor-memory accumulator in tile order (bit-identical from
// run to run).  With one CTA per slice only as many SMs as slices stream; each keeps ten
// 16 KB ring slots in flight.
// Warps: 0-7 row warps in two groups taking alternate tiles (group g = warp / 4 owns TMEM
// lanes 32 (warp % 4) + [0, 32) of its own S and H buffers); 8 and 10 producers, each with
// its own five-slot TMA ring (warp 8: Q_t in pass 1, then A_t in pass 2; warp 10: V_t): a Q
// slot is free again as soon as S_t has read it, so the Q loads run further ahead of their
// use than a shared [Q | V] slot, which only the later W MMA frees, would allow; 9 issues
// S_t (and the pass-2 H MMAs), 11 issues the W MMAs: a tcgen05.mma holds its issuing thread
// until the tensor pipe takes it (about 48 cycles at N = 64, 52 at N = 80), so one thread
// issuing both kinds (12 per tile) between its waits set the tile rate.  Pass 1 is then bound
// by the bytes in flight: the deepest rings that fit shared memory (five slots each, with two
// row-warp groups; a third group, which leaves room for four slots only, was slower, and so
// was Delta as an MMA of its own over a smaller ones block).  Launched with programmatic
// stream serialization: the setup overlaps the previous kernel, global memory comes after
// griddepcontrol.wait.
// Every wait is bounded; one that gives up sets bit 0 of this kernel's error word and the
// CTA drains what it has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_stream_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128, kD = 64, kMP = 64;
constexpr int kNG = 2;                 // row-warp groups, taking tiles t = g (mod kNG)
constexpr int kRowWarps = 4 * kNG;
constexpr int kThreads = 32 * (kRowWarps + 4);
constexpr int kWarpProducer = kRowWarps, kWarpMma = kRowWarps + 1, kWarpProducerV = kRowWarps + 2,
              kWarpMmaW = kRowWarps + 3;
constexpr int kSlots = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileB = kT * 64 * 2;   // a [128][64] bf16 tile (16 KB)

constexpr int kImgB = kMP * kD * 2;
// shared memory (an MN-major M = 128 operand reads an unused second 64-row block 16 KB on:
// the last A tile's is the first Q slot)
constexpr int kOffA = 0;                             // A tiles of the row-warp groups
constexpr int kOffQRing = kOffA + kNG * kTileB;      // Q ring: Q_t in pass 1, then A_t in pass 2
constexpr int kOffVRing = kOffQRing + kSlots * kTileB;  // V ring; in pass 2 the H staging (4 KB per row warp)
constexpr int kOffOnes = kOffVRing + kSlots * kTileB;   // [128][64] bf16 ones: the second block of [V | 1]
constexpr int kOffU = kOffOnes + kTileB;             // U [64][64]
constexpr int kOffW = kOffU + kImgB;                 // W' image [64][64]
constexpr int kOffStage = kOffVRing;
constexpr int kOffBar = kOffW + kImgB;
constexpr int kBars = 4 * kSlots + 4 * kNG + 2 * kNG * 2 + 6;
constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kOffStage + kRowWarps * 4096 <= kOffOnes, "pass-2 staging inside the V ring");
// tensor memory: pass 1 S_g at 64 g and [W | Delta] after them; pass 2 (W read out by then)
// H of group g, buffer b at 64 (2 g + b)
constexpr uint32_t kColS = 0, kColW = 64 * kNG, kColDelta = kColW + 64, kColH = 0;
static_assert(kColDelta + 16 <= 512 && 64 * 2 * kNG <= 512, "tensor memory columns");

struct StParams {
    int heads, n, m, tiles;
    float c;  // scale * log2(e)
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}
__device__ __forceinline__ uint4 pack8(const float *x, float r) {
    return make_uint4(pack2(x[0] * r, x[1] * r), pack2(x[2] * r, x[3] * r), pack2(x[4] * r, x[5] * r),
                      pack2(x[6] * r, x[7] * r));
}

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_stream_error, 1u);
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
anchor_stream_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap ta_st,
                     const __grid_constant__ CUtensorMap ta_ld, const __grid_constant__ CUtensorMap th,
                     const StParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *full = bars, *empty = full + kSlots, *vfull = empty + kSlots, *vempty = vfull + kSlots;
    uint64_t *s_full = vempty + kSlots, *s_empty = s_full + kNG, *a_full = s_empty + kNG, *a_empty = a_full + kNG;
    uint64_t *h_full = a_empty + kNG, *h_empty = h_full + 2 * kNG;  // [2 g + b]
    uint64_t *u_full = h_empty + 2 * kNG, *w_full = u_full + 1, *wp_full = u_full + 2, *mma_done = u_full + 3;
    uint64_t *mma_done_w = u_full + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x;
    const int h = slice % p.heads;
    const int T = p.tiles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
            mbar_init(vfull + i, 1);
            mbar_init(vempty + i, 1);
        }
        for (int g = 0; g < kNG; ++g) {
            mbar_init(s_full + g, 1);
            mbar_init(s_empty + g, 4);
            mbar_init(a_full + g, 4);
            mbar_init(a_empty + g, 1);
        }
        for (int i = 0; i < 2 * kNG; ++i) {
            mbar_init(h_full + i, 1);
            mbar_init(h_empty + i, 4);
        }
        mbar_init(u_full, 1);
        mbar_init(w_full, 1);
        mbar_init(wp_full, kRowWarps);
        mbar_init(mma_done, 1);
        mbar_init(mma_done_w, 1);
        fence_mbar_init();
    }
    if (warp < kRowWarps) {  // the ones block
        const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = threadIdx.x; i < kTileB / 16; i += 32 * kRowWarps) reinterpret_cast<uint4 *>(sm + kOffOnes)[i] = ones;
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t sbase = smem_u32(sm);
    // launched with programmatic stream serialization: the setup above may run while the
    // previous kernel in the stream finishes; global memory only from here on
    grid_dependency_wait();
    grid_dependents_launch();

    if (warp == kWarpProducer) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tu);
            tma_prefetch_desc(&ta_ld);
            const uint64_t pol_once = policy_evict_first(), pol_keep = policy_evict_last();
            mbar_arrive_expect_tx(u_full, kImgB);
            tma_load_3d(sm + kOffU, &tu, u_full, 0, 0, h, pol_keep);
            int issued = 0;
            for (int seq = 0; seq < 2 * T; ++seq) {
                const int s = seq % kSlots;
                if (seq >= kSlots && !bwait(empty + s, (uint32_t)(((seq / kSlots) - 1) & 1), p.wait_ns)) break;
                uint8_t *st = sm + kOffQRing + s * kTileB;
                if (seq < T) {
                    mbar_arrive_expect_tx(full + s, kTileB);
                    tma_load_3d(st, &tq, full + s, 0, seq * kT, slice, pol_once);
                } else {
                    // pass 2: every A tile has been stored (the row warps finish their stores
                    // before they arrive on wp_full)
                    if (seq == T && !bwait(wp_full, 0u, p.wait_ns)) break;
                    mbar_arrive_expect_tx(full + s, kTileB);
                    tma_load_3d(st, &ta_ld, full + s, 0, (seq - T) * kT, slice, pol_once);
                }
                ++issued;
            }
            for (int s = 0; s < kSlots; ++s) {
                const int loads = issued > s ? (issued - s + kSlots - 1) / kSlots : 0;
                if (loads > 0) bwait(full + s, (uint32_t)((loads - 1) & 1), p.wait_ns);
            }
            bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpProducerV) {
        if (lane == 0) {
            tma_prefetch_desc(&tv);
            const uint64_t pol_once = policy_evict_first();
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int s = t % kSlots;
                if (t >= kSlots && !bwait(vempty + s, (uint32_t)(((t / kSlots) - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(vfull + s, kTileB);
                tma_load_3d(sm + kOffVRing + s * kTileB, &tv, vfull + s, 0, t * kT, slice, pol_once);
                ++issued;
            }
            for (int s = 0; s < kSlots; ++s) {
                const int loads = issued > s ? (issued - s + kSlots - 1) / kSlots : 0;
                if (loads > 0) bwait(vfull + s, (uint32_t)((loads - 1) & 1), p.wait_ns);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);       // S = Q U^T
            const uint32_t idH = idesc_bf16_f32(kT, kD, false, true);         // H = A W'
            const uint64_t udesc = smem_desc_sw128(sbase + kOffU, 16, 1024);
            const uint64_t wdesc = smem_desc_sw128(sbase + kOffW, kMP * 128, 1024);
            bool ok = bwait(u_full, 0u, p.wait_ns);
            // pass 1: S_t as soon as Q_t is in and its group has read S_{t-2}
            for (int t = 0; t < T && ok; ++t) {
                const int s = t % kSlots, g = t % kNG, k = t / kNG;
                if (!bwait(full + s, (uint32_t)((t / kSlots) & 1), p.wait_ns)) { ok = false; break; }
                if (k >= 1 && !bwait(s_empty + g, (uint32_t)((k - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(sbase + kOffQRing + s * kTileB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16(tmem + kColS + g * 64, qdesc + (uint64_t)(kk * 2), udesc + (uint64_t)(kk * 2), idS,
                              kk > 0 ? 1u : 0u);
                umma_commit(s_full + g);
                umma_commit(empty + s);  // Q_t has been read
            }
            // pass 2: H_t = A_t W'
            ok = ok && bwait(wp_full, 0u, p.wait_ns);
            for (int t = 0; t < T && ok; ++t) {
                // H buffer (g, b) of tile t = g + kNG k: b = k & 1, its use number k >> 1
                const int seq = T + t, s = seq % kSlots, k = t / kNG, hb = 2 * (t % kNG) + (k & 1), u = k >> 1;
                if (!bwait(full + s, (uint32_t)((seq / kSlots) & 1), p.wait_ns)) { ok = false; break; }
                if (u >= 1 && !bwait(h_empty + hb, (uint32_t)((u - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint64_t adesc = smem_desc_sw128(sbase + kOffQRing + s * kTileB, 16, 1024);
#pragma unroll
                for (int kj = 0; kj < kMP / 16; ++kj)
                    umma_bf16(tmem + kColH + hb * 64, adesc + (uint64_t)(kj * 2), wdesc + (uint64_t)(kj * 128), idH,
                              kj > 0 ? 1u : 0u);
                umma_commit(h_full + hb);
                umma_commit(empty + s);
            }
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpMmaW) {
        if (lane == 0) {
            const uint32_t idWD = idesc_bf16_f32(kT, kD + 16, true, true);    // [W | Delta] += A^T [V | 1]
            bool ok = true;
            for (int t = 0; t < T && ok; ++t) {
                const int s = t % kSlots, g = t % kNG;
                if (!bwait(a_full + g, (uint32_t)((t / kNG) & 1), p.wait_ns) ||
                    !bwait(vfull + s, (uint32_t)((t / kSlots) & 1), p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t va = sbase + kOffVRing + s * kTileB;
                const uint64_t adesc = smem_desc_sw128(sbase + kOffA + g * kTileB, kTileB, 1024);
                // [V | 1]: the ones block is the B operand's second 64-column block
                const uint64_t vdesc = smem_desc_sw128(va, sbase + kOffOnes - va, 1024);
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + kColW, adesc + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), idWD,
                              (t > 0 || kt > 0) ? 1u : 0u);
                umma_commit(a_empty + g);
                umma_commit(vempty + s);
            }
            if (ok) umma_commit(w_full);
            umma_commit(mma_done_w);
            bwait(mma_done_w, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        const int g = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        uint8_t *sA = sm + kOffA + g * kTileB;
        const uint64_t pol_a = policy_evict_last(), pol_out = policy_evict_first();
        bool ok = true;
        float v[64];
        for (int t = g, k = 0; t < T && ok; t += kNG, ++k) {
            if (!bwait(s_full + g, (uint32_t)(k & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColS + g * 64, v);
            tmem_ld32(trow + kColS + g * 64 + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty + g);
            // A_ij = 2^(c S_ij - max_j c S_ij) / sum; anchors >= m get 0; tokens >= n a zero row
            const float z = rowops::softmax64_unnormalised(v, p.m, p.c);
            rowops::scale64(v, t * kT + row < p.n ? 1.f / z : 0.f);
            // the group's A buffer: the W MMA of its previous tile has read it, and so has
            // this warp's TMA store of it
            if (k >= 1 && !bwait(a_empty + g, (uint32_t)((k - 1) & 1), p.wait_ns)) { ok = false; break; }
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) *reinterpret_cast<uint4 *>(sA + sw_off(row, c8, kT)) = pack8(v + 8 * c8);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(a_full + g);
                if (t * kT + q * 32 < p.n) {
                    tma_store_3d(&ta_st, sA + q * 32 * 128, 0, t * kT + q * 32, slice, pol_a);
                    bulk_commit_group();
                }
            }
        }
        // every A store of this warp is complete and visible to the pass-2 loads
        if (lane == 0) {
            bulk_wait_group0();
            fence_proxy_async_global();
        }
        __syncwarp();
        // W' = W / Delta (anchor j = row: warps 0 and 1)
        ok = ok && bwait(w_full, 0u, p.wait_ns);
        if (ok) {
            if (warp < 2) {
                tc_fence_after();
                float w[64], dl[32];
                tmem_ld32(trow + kColW, w);
                tmem_ld32(trow + kColW + 32, w + 32);
                tmem_ld32(trow + kColDelta, dl);
                tmem_ld_wait();
                const float rinv = dl[0] != 0.f ? 1.f / dl[0] : 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm + kOffW + sw_off(row, c8, kMP)) = pack8(w + 8 * c8, rinv);
                fence_proxy_async_smem();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(wp_full);
        }
        // pass 2: H tiles out
        uint8_t *stage = sm + kOffStage + warp * 4096;
        for (int t = g, k = 0; t < T && ok; t += kNG, ++k) {
            const int hb = 2 * g + (k & 1);
            if (!bwait(h_full + hb, (uint32_t)((k >> 1) & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColH + hb * 64, v);
            tmem_ld32(trow + kColH + hb * 64 + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(h_empty + hb);
                bulk_wait_group_read0();  // the last store has read the staging
            }
            __syncwarp();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(stage + sw_off(lane, c8, 32)) = pack8(v + 8 * c8);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && t * kT + q * 32 < p.n) {
                tma_store_3d(&th, stage, 0, t * kT + q * 32, slice, pol_out);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool stream_supported(const Problem &p) { return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1; }

size_t stream_workspace(const Problem &p) { return (size_t)p.slices() * p.n * kD * 2; }

cudaError_t launch_stream(const Problem &p, void *workspace, cudaStream_t stream) {
    CUtensorMap tq, tv, tu, ta_st, ta_ld, th;
    const long long S = p.slices();
    if (!make_bf16_map(&tq, p.Q, kD, p.n, S, kT) || !make_bf16_map(&tv, p.V, kD, p.n, S, kT) ||
        !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP) || !make_bf16_map(&ta_st, workspace, kMP, p.n, S, 32) ||
        !make_bf16_map(&ta_ld, workspace, kMP, p.n, S, kT) || !make_bf16_map(&th, p.H, kD, p.n, S, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(anchor_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    StParams sp;
    sp.heads = p.heads;
    sp.n = p.n;
    sp.m = p.m;
    sp.tiles = (p.n + kT - 1) / kT;
    sp.c = p.scale * 1.4426950408889634f;
    sp.wait_ns = 2000000000ull;
    return launch_pdl(anchor_stream_kernel, dim3((unsigned)S), dim3(kThreads), kSmem, stream, tq, tv, tu, ta_st, ta_ld,
                      th, sp);
}

cudaError_t stream_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_stream_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

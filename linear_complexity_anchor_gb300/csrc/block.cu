// Block front end of the anchor attention: the per-head queries and values are projections of
// the token embeddings (an AnchorFormer layer puts the anchor attention where a ViT block has
// its self-attention), computed inside the kernel so that X is read once and Q, V never reach
// global memory:
//   Q = X Wq_h^T,  V = X Wv_h^T            (X [n][dm], Wq_h, Wv_h [d][dm])
//   A = rowsoftmax(scale Q U_h^T),  W' = Delta^{-1} (A^T V),  H = A W'
// (pith.science verdict on arXiv 2505.16463: "key_machinery", the referee summary of Eq. 11/12;
// the arXiv abstract, where the anchors are weights of a trainable layer).
//
// One CTA per (batch, head) slice of up to 256 tokens (two 128-token tiles), d = 64, m <= 64,
// two CTAs per SM so that one CTA's projection overlaps the other's anchor steps.  Warps:
//   0-3  row warps: warp w owns TMEM lanes 32w..32w+31 (tokens of a tile, or anchors);
//        they move the projections out of tensor memory into bf16 operand tiles, take the
//        row softmax, form the W' image and store H
//   4    producer: TMA loads of U and of the projection operands (a two-stage ring of
//        [X tile 0 | X tile 1 | Wq_h rows | Wv_h rows] 64-column chunks)
//   5    MMA issuer (one thread): [Q|V]_t += X_t [Wq_h; Wv_h]^T (M = 128, N = 128, K = dm),
//        S_t = Q_t U^T, [W | Delta] += A_t^T [V_t | 1], H_t = A_t W'
// After the projection the steps go tile by tile (tile 0's S and W MMAs run while the row
// warps convert and take the softmax of tile 1).
// Tensor memory (256 columns): projections P_t = [Q_t | V_t] at 128 t; then S_t and H_t at
// 64 t, W at 128, Delta at 192.  Every wait is bounded; a wait that gives up sets bit 0 of the
// block error word and the CTA drains what it has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_block_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128;           // tokens per tile (MMA M)
constexpr int kD = 64;            // head dimension
constexpr int kMP = 64;           // anchors, padded
constexpr int kKC = 64;           // embedding columns per ring stage
constexpr int kThreads = 192;
constexpr int kWarpProducer = 4, kWarpMma = 5;
constexpr uint32_t kTmemCols = 256;

// shared memory (bytes from a 1024-aligned base)
constexpr int kTileB = kT * 64 * 2;                 // one 128 x 64 bf16 tile: 16 KB
constexpr int kStageB = 3 * kTileB;                 // X tile 0 | X tile 1 | Wq rows | Wv rows
constexpr int kRingB = 2 * kStageB;                 // 96 KB
// after the projection the ring holds: Q_t / A_t at t * 16 KB, V_t (then the H_t staging) at
// 32 KB + t * 16 KB, the ones block [128][64] (16 KB) and then the W' image at 64 KB
constexpr int kOffV = 2 * kTileB;
constexpr int kOffW = 4 * kTileB;
// The same kernel runs the plain forward on short slices (kProj = false): Q and V then arrive
// by TMA straight into the tiles at 0 and 32 KB, and shared memory ends after the ones block.
template <bool kProj> struct BlockLayout {
    static constexpr int kOffU = kProj ? kRingB : 5 * kTileB;   // U [64][64] bf16, 8 KB
    static constexpr int kOffBar = kOffU + kMP * kD * 2;
    static constexpr int kSmem = kOffBar + 20 * 8 + 16 + 1024;  // + alignment slack
};
constexpr int kBars = 20;

struct BlockParams {
    int heads, n, m, dm, tiles;
    float c;             // scale * log2(e)
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8(const float *x, float r) {
    return make_uint4(pack2(x[0] * r, x[1] * r), pack2(x[2] * r, x[3] * r), pack2(x[4] * r, x[5] * r),
                      pack2(x[6] * r, x[7] * r));
}


__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bounded wait for the phase of `bar` with parity `par`; false (and bit 0) when it gives up
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_block_error, 1u);
            return false;
        }
    }
    return true;
}

template <bool kProj>
__global__ void __launch_bounds__(kThreads, 2)
anchor_block_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap twq,
                    const __grid_constant__ CUtensorMap twv, const __grid_constant__ CUtensorMap tu,
                    const __grid_constant__ CUtensorMap th, const BlockParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    using LY = BlockLayout<kProj>;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::kOffBar);
    uint64_t *full = bars + 0, *empty = bars + 2;
    uint64_t *proj_done = bars + 4, *u_full = bars + 5, *w_full = bars + 6, *wp_full = bars + 7;
    uint64_t *mma_done = bars + 8;
    // per token tile t: qv_full + t (Q_t, V_t written), s_full + t, a_full + t, h_full + t
    uint64_t *qv_full = bars + 9, *s_full = bars + 11, *a_full = bars + 13, *h_full = bars + 15;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x;
    const int b = slice / p.heads, h = slice - b * p.heads;
    const int T = p.tiles;
    const int KC = p.dm / kKC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        mbar_init(proj_done, 1);
        mbar_init(u_full, 1);
        mbar_init(w_full, 1);
        mbar_init(wp_full, 4);
        mbar_init(mma_done, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(qv_full + t, 4);
            mbar_init(s_full + t, 1);
            mbar_init(a_full + t, 4);
            mbar_init(h_full + t, 1);
        }
        fence_mbar_init();
    }
    if (warp == kWarpMma) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t sbase = smem_u32(sm);
    // launched with programmatic stream serialization: global memory only from here on
    grid_dependency_wait();
    grid_dependents_launch();

    if (warp == kWarpProducer) {
        if (lane == 0) {
            tma_prefetch_desc(&tx);
            tma_prefetch_desc(&twq);
            tma_prefetch_desc(&twv);
            tma_prefetch_desc(&tu);
            const uint64_t pol_keep = policy_evict_last(), pol_x = policy_evict_normal();
            mbar_arrive_expect_tx(u_full, kMP * kD * 2);
            tma_load_3d(sm + LY::kOffU, &tu, u_full, 0, 0, h, pol_keep);
            int issued = 0;
            if constexpr (kProj) {
                for (int kc = 0; kc < KC; ++kc) {
                    const int s = kc & 1;
                    if (kc >= 2 && !bwait(empty + s, ((kc >> 1) + 1) & 1u, p.wait_ns)) break;
                    uint8_t *st = sm + s * kStageB;
                    mbar_arrive_expect_tx(full + s, (uint32_t)(T * kTileB + kTileB));
                    for (int t = 0; t < T; ++t) tma_load_3d(st + t * kTileB, &tx, full + s, kc * kKC, t * kT, b, pol_x);
                    tma_load_3d(st + 2 * kTileB, &twq, full + s, kc * kKC, 0, h, pol_keep);
                    tma_load_3d(st + 2 * kTileB + kTileB / 2, &twv, full + s, kc * kKC, 0, h, pol_keep);
                    ++issued;
                }
            } else {  // Q_t and V_t of the slice (tx: the Q map, twq: the V map), one barrier per tile
                for (int t = 0; t < T; ++t) {
                    mbar_arrive_expect_tx(full + t, 2 * kTileB);
                    tma_load_3d(sm + t * kTileB, &tx, full + t, 0, t * kT, slice, pol_x);
                    tma_load_3d(sm + kOffV + t * kTileB, &twq, full + t, 0, t * kT, slice, pol_x);
                }
                issued = T;
            }
            // the last loads of each stage (each tile) and of U have landed before the CTA leaves
            for (int s = 0; s < 2; ++s) {
                const int loads = kProj ? (issued > s ? (issued - s + 1) / 2 : 0) : (issued > s ? 1 : 0);
                if (loads > 0) bwait(full + s, (uint32_t)((loads - 1) & 1), p.wait_ns);
            }
            bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint32_t kIdP = idesc_bf16_f32(kT, 2 * kD, false, false);  // [Q|V] += X [Wq; Wv]^T
            const uint32_t kIdS = idesc_bf16_f32(kT, kMP, false, false);     // S = Q U^T
            const uint32_t kIdWD = idesc_bf16_f32(kT, kD + 16, true, true);  // [W | Delta] += A^T [V | 1]
            const uint32_t kIdH = idesc_bf16_f32(kT, kD, false, true);       // H = A W'
            bool ok = true;
            for (int kc = 0; kProj && kc < KC; ++kc) {
                const int s = kc & 1;
                if (!bwait(full + s, (uint32_t)((kc >> 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st = sbase + s * kStageB;
                const uint64_t wdesc = smem_desc_sw128(st + 2 * kTileB, 16, 1024);
                for (int t = 0; t < T; ++t) {
                    const uint64_t xdesc = smem_desc_sw128(st + t * kTileB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk)
                        umma_bf16(tmem + t * 128, xdesc + (uint64_t)(kk * 2), wdesc + (uint64_t)(kk * 2), kIdP,
                                  (kc > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(empty + s);
            }
            if (kProj && ok) umma_commit(proj_done);
            // tile by tile, so that tile 0's S and W run while the row warps work on tile 1
            ok = ok && bwait(u_full, 0u, p.wait_ns);
            const uint64_t udesc = smem_desc_sw128(sbase + LY::kOffU, 16, 1024);
            for (int t = 0; t < T && ok; ++t) {
                // the tile's Q and V: written by the row warps from the projection, or loaded
                if (!bwait(kProj ? qv_full + t : full + t, 0u, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(sbase + t * kTileB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16(tmem + t * 64, qdesc + (uint64_t)(kk * 2), udesc + (uint64_t)(kk * 2), kIdS,
                              kk > 0 ? 1u : 0u);
                umma_commit(s_full + t);
            }
            // the ones block is written (by the row warps, before qv_full + 0)
            if (!kProj) ok = ok && bwait(qv_full, 0u, p.wait_ns);
            for (int t = 0; t < T && ok; ++t) {
                if (!bwait(a_full + t, 0u, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                // A^T as the M = 128 operand: anchors 64..127 read the next 16 KB (never used);
                // [V | 1]: the ones block is the B operand's second 64-column block
                const uint32_t va = sbase + kOffV + t * kTileB;
                const uint64_t adesc = smem_desc_sw128(sbase + t * kTileB, kTileB, 1024);
                const uint64_t vdesc = smem_desc_sw128(va, sbase + kOffW - va, 1024);
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + 128, adesc + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), kIdWD,
                              (t > 0 || kt > 0) ? 1u : 0u);
            }
            if (ok) umma_commit(w_full);
            ok = ok && bwait(wp_full, 0u, p.wait_ns);
            if (ok) {
                tc_fence_after();
                const uint64_t wdesc = smem_desc_sw128(sbase + kOffW, kMP * 128, 1024);
                for (int t = 0; t < T; ++t) {
                    const uint64_t adesc = smem_desc_sw128(sbase + t * kTileB, 16, 1024);
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16(tmem + t * 64, adesc + (uint64_t)(kj * 2), wdesc + (uint64_t)(kj * 128), kIdH,
                                  kj > 0 ? 1u : 0u);
                    umma_commit(h_full + t);
                }
            }
            // every MMA issued has completed before the CTA leaves
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        const int row = warp * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
        if (!kProj) {  // the ones block of [V | 1] ([128][64] bf16 ones, 16 KB)
            const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
            for (int i = row; i < kTileB / 16; i += 128) reinterpret_cast<uint4 *>(sm + kOffW)[i] = ones;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qv_full);
        }
        if (kProj) ok = bwait(proj_done, 0u, p.wait_ns);
        if (kProj && ok) {
            tc_fence_after();
            float v[64];
            for (int t = 0; t < T; ++t) {
                // Q_t and V_t rows as bf16 K-major / MN-major operand tiles (same swizzled layout)
                tmem_ld32(trow + t * 128, v);
                tmem_ld32(trow + t * 128 + 32, v + 32);
                tmem_ld_wait();
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm + t * kTileB + sw_off(row, c8, kT)) = pack8(v + 8 * c8, 1.f);
                tmem_ld32(trow + t * 128 + 64, v);
                tmem_ld32(trow + t * 128 + 96, v + 32);
                tmem_ld_wait();
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm + kOffV + t * kTileB + sw_off(row, c8, kT)) = pack8(v + 8 * c8, 1.f);
                if (t == 0) {  // the ones block of [V | 1] ([128][64] bf16 ones, 16 KB)
                    const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
                    for (int i = row; i < kTileB / 16; i += 128) reinterpret_cast<uint4 *>(sm + kOffW)[i] = ones;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(qv_full + t);
            }
        }
        for (int t = 0; t < T && ok; ++t) {
            if (!bwait(s_full + t, 0u, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            float v[64];
            tmem_ld32(trow + t * 64, v);
            tmem_ld32(trow + t * 64 + 32, v + 32);
            tmem_ld_wait();
            // A_ij = 2^(c S_ij - max_j c S_ij) / sum; anchors >= m get 0; tokens >= n a zero row
            const float z = rowops::softmax64_unnormalised(v, p.m, p.c);
            rowops::scale64(v, t * kT + row < p.n ? 1.f / z : 0.f);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + t * kTileB + sw_off(row, c8, kT)) = pack8(v + 8 * c8, 1.f);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + t);
        }
        ok = ok && bwait(w_full, 0u, p.wait_ns);
        if (ok) {
            if (warp < 2) {  // lanes 0..63: anchor j = row; W'_j = W_j / Delta_j (0 if Delta_j = 0)
                tc_fence_after();
                float w[64], dl[32];
                tmem_ld32(trow + 128, w);
                tmem_ld32(trow + 160, w + 32);
                tmem_ld32(trow + 192, dl);
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
        if (ok) {
            const uint64_t pol_out = policy_evict_first();
            float v[64];
            for (int t = 0; t < T; ++t) {
                if (!bwait(h_full + t, 0u, p.wait_ns)) break;
                tc_fence_after();
                tmem_ld32(trow + t * 64, v);
                tmem_ld32(trow + t * 64 + 32, v + 32);
                tmem_ld_wait();
                // staged over V_t (free since the W MMAs; the H MMA of the other tile may still
                // be reading A and W')
                uint8_t *stage = sm + kOffV + t * kTileB + warp * 4096;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(stage + sw_off(lane, c8, 32)) = pack8(v + 8 * c8, 1.f);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && t * kT + warp * 32 < p.n) {
                    tma_store_3d(&th, stage, 0, t * kT + warp * 32, slice, pol_out);
                    bulk_commit_group();
                }
            }
            if (lane == 0) bulk_wait_group0();
            tc_fence_before();
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool block_supported(const BlockProblem &p) {
    return p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1 && p.n <= 2 * kT && p.dm >= kKC && p.dm % kKC == 0;
}

cudaError_t launch_block(const BlockProblem &p, cudaStream_t stream) {
    CUtensorMap tx, twq, twv, tu, th;
    const long long slices = (long long)p.B * p.heads;
    if (!make_bf16_map(&tx, p.X, p.dm, p.n, p.B, kT) || !make_bf16_map(&twq, p.Wq, p.dm, kD, p.heads, kD) ||
        !make_bf16_map(&twv, p.Wv, p.dm, kD, p.heads, kD) || !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP) ||
        !make_bf16_map(&th, p.H, kD, p.n, slices, 32))
        return cudaErrorInvalidValue;
    constexpr int kSmem = BlockLayout<true>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(anchor_block_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    BlockParams bp;
    bp.heads = p.heads;
    bp.n = p.n;
    bp.m = p.m;
    bp.dm = p.dm;
    bp.tiles = (p.n + kT - 1) / kT;
    bp.c = p.scale * 1.4426950408889634f;
    bp.wait_ns = 2000000000ull;
    return launch_pdl(anchor_block_kernel<true>, dim3((unsigned)slices), dim3(kThreads), kSmem, stream, tx, twq, twv, tu,
                      th, bp);
}

bool short_supported(const Problem &p) {
    return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1 && p.n <= 2 * kT;
}

// The plain forward on slices of up to 256 tokens: the same kernel with Q and V loaded.
cudaError_t launch_short(const Problem &p, cudaStream_t stream) {
    CUtensorMap tq, tv, tu, th;
    const long long slices = p.slices();
    if (!make_bf16_map(&tq, p.Q, kD, p.n, slices, kT) || !make_bf16_map(&tv, p.V, kD, p.n, slices, kT) ||
        !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP) || !make_bf16_map(&th, p.H, kD, p.n, slices, 32))
        return cudaErrorInvalidValue;
    constexpr int kSmem = BlockLayout<false>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(anchor_block_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    BlockParams bp;
    bp.heads = p.heads;
    bp.n = p.n;
    bp.m = p.m;
    bp.dm = kKC;
    bp.tiles = (p.n + kT - 1) / kT;
    bp.c = p.scale * 1.4426950408889634f;
    bp.wait_ns = 2000000000ull;
    return launch_pdl(anchor_block_kernel<false>, dim3((unsigned)slices), dim3(kThreads), kSmem, stream, tq, tv, tq, tu,
                      th, bp);
}

cudaError_t block_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_block_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_block_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

// Masked (causal) variant of the anchor-attention forward on the tensor cores (bf16 operands,
// fp32 accumulators in tensor memory) for d = 64 and m <= 64, any n.  Token i's anchor
// summaries include only tokens j <= i (one of the inferences of the pith.science verdict on
// arXiv 2505.16463: A can be masked against later tokens without giving up the O(mn) cost):
//   Delta^(i)_l = sum_{j<=i} A[j][l],  W^(i)_l = sum_{j<=i} A[j][l] v_j,
//   H[i] = sum_l A[i][l] W^(i)_l / Delta^(i)_l   (0 for an anchor with Delta^(i)_l = 0).
//
// One CTA per (batch, head) slice walks the slice's 128-token tiles in order, keeping the
// summaries of the tiles before (W_pre in tensor memory, Delta_pre in shared memory).  Per
// tile t, with B[i][l] = A[i][l] / Delta^(i)_l:
//   S_t = Q_t U^T, A_t = softmax (row warps)
//   C_t = L A_t, L the lower-triangular [128][128] ones: the running column sums inside the
//        tile, so Delta^(i) = Delta_pre + C_t[i] (row warps, which then form B_t)
//   P_t = B_t A_t^T, masked to j <= i by the row warps
//   H_t = B_t W_pre + P_t V_t
//   W_pre += A_t^T V_t, Delta_pre += the tile's column sums (the last row of C_t)
// The sums over j use the bf16 A_t in every place (C_t, P_t, W_pre), so Delta and W stay
// consistent; B on the i side is formed from the fp32 A.  Warps: 0-3 row warps (TMEM lanes
// 32w..32w+31: tokens, or anchors for the W_pre image; a tile's H goes out, and the next W_pre
// image is written, while the next tile's C runs), 4 producer (TMA ring of [Q_t | V_t]),
// 5 MMA issuer.  Sums run in a fixed order: results are bit-identical from run to run.  Every
// wait is bounded; one that gives up sets bit 0 of this kernel's error word and the CTA drains
// what it has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_causal_tc_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128, kD = 64, kMP = 64;
constexpr int kThreads = 192;
constexpr int kWarpProducer = 4, kWarpMma = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileB = kT * 64 * 2;    // a [128][64] bf16 tile (16 KB)
constexpr int kSlotB = 2 * kTileB;     // Q_t | V_t
constexpr int kImgB = kMP * kD * 2;    // [64][64] bf16 (8 KB)
// shared memory
constexpr int kOffU = 2 * kSlotB;              // U [64][64]
constexpr int kOffL = kOffU + kImgB;           // L [128][128] (two 64-column blocks)
constexpr int kOffA = kOffL + 2 * kTileB;      // A_t [128][64]; its unused second M block (W MMA) is B_t
constexpr int kOffB = kOffA + kTileB;          // B_t [128][64]
constexpr int kOffP = kOffB + kTileB;          // P_t [128][128]
constexpr int kOffWI = kOffP + 2 * kTileB;     // W_pre image [64][64]
constexpr int kOffDP = kOffWI + kImgB;         // Delta_pre [2][64] fp32
constexpr int kOffBar = kOffDP + 512;
constexpr int kBars = 24;
constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
// tensor memory columns
constexpr uint32_t kColS0 = 0, kColC = 128, kColP = 192, kColH = 320, kColW = 384;

struct CtcParams {
    int heads, n, m, tiles;
    float c;   // scale * log2(e)
    __nv_bfloat16 *H;
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

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_causal_tc_error, 1u);
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
anchor_causal_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                        const __grid_constant__ CUtensorMap tu, const CtcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *full = bars + 0, *empty = bars + 2, *s_full = bars + 4, *s_empty = bars + 6;
    uint64_t *u_full = bars + 8, *a_full = bars + 9, *c_full = bars + 10, *b_full = bars + 11;
    uint64_t *p_full = bars + 12, *pm_full = bars + 13, *h_full = bars + 14, *h_empty = bars + 15;
    uint64_t *w_full = bars + 16, *wi_full = bars + 17, *mma_done = bars + 18, *dp_full = bars + 19;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);
    float *sDP = reinterpret_cast<float *>(sm + kOffDP);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x;
    const int h = slice % p.heads;
    const int T = p.tiles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
            mbar_init(s_full + i, 1);
            mbar_init(s_empty + i, 4);
        }
        mbar_init(u_full, 1);
        mbar_init(a_full, 4);
        mbar_init(c_full, 1);
        mbar_init(b_full, 4);
        mbar_init(p_full, 1);
        mbar_init(pm_full, 4);
        mbar_init(h_full, 1);
        mbar_init(h_empty, 4);
        mbar_init(w_full, 1);
        mbar_init(wi_full, 4);
        mbar_init(mma_done, 1);
        mbar_init(dp_full, 4);
        fence_mbar_init();
    }
    if (warp < 4) {  // row warps: L[i][j] = 1 for j <= i (row i = this thread), Delta_pre = 0
        const int row = threadIdx.x;
        const uint32_t one = 0x3F80u;
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
            uint32_t w4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = c8 * 8 + 2 * q;
                w4[q] = (j <= row ? one : 0u) | ((j + 1 <= row ? one : 0u) << 16);
            }
            *reinterpret_cast<uint4 *>(sm + kOffL + sw_off(row, c8, kT)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        if (row < 64) sDP[row] = 0.f;
        fence_proxy_async_smem();
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
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tu);
            const uint64_t pol_keep = policy_evict_last(), pol_once = policy_evict_first();
            mbar_arrive_expect_tx(u_full, kImgB);
            tma_load_3d(sm + kOffU, &tu, u_full, 0, 0, h, pol_keep);
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int s = t & 1;
                if (t >= 2 && !bwait(empty + s, (uint32_t)(((t >> 1) - 1) & 1), p.wait_ns)) break;
                uint8_t *st = sm + s * kSlotB;
                mbar_arrive_expect_tx(full + s, 2 * kTileB);
                tma_load_3d(st, &tq, full + s, 0, t * kT, slice, pol_once);
                tma_load_3d(st + kTileB, &tv, full + s, 0, t * kT, slice, pol_once);
                ++issued;
            }
            for (int s = 0; s < 2; ++s) {
                const int loads = issued > s ? (issued - s + 1) / 2 : 0;
                if (loads > 0) bwait(full + s, (uint32_t)((loads - 1) & 1), p.wait_ns);
            }
            bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);   // [tokens x anchors], K = d
            const uint32_t idC = idesc_bf16_f32(kT, kMP, false, true);    // L A: K = tokens
            const uint32_t idP = idesc_bf16_f32(kT, kT, false, false);    // B A^T: [tokens x tokens], K = anchors
            const uint32_t idH = idesc_bf16_f32(kT, kD, false, true);     // [tokens x d]
            const uint32_t idW = idesc_bf16_f32(kT, kD, true, true);      // A^T V: anchors x d, K = tokens
            const uint64_t udesc = smem_desc_sw128(sbase + kOffU, 16, 1024);
            const uint64_t ldesc = smem_desc_sw128(sbase + kOffL, 16, 1024);
            const uint64_t amn = smem_desc_sw128(sbase + kOffA, kTileB, 1024);   // A_t, MN-major
            const uint64_t ak = smem_desc_sw128(sbase + kOffA, 16, 1024);        // A_t, K-major
            const uint64_t bk = smem_desc_sw128(sbase + kOffB, 16, 1024);        // B_t, K-major
            const uint64_t pk = smem_desc_sw128(sbase + kOffP, 16, 1024);        // P_t, K-major
            const uint64_t wim = smem_desc_sw128(sbase + kOffWI, kMP * 128, 1024);  // W_pre image, MN-major
            bool ok = bwait(u_full, 0u, p.wait_ns);
            auto issue_s = [&](int t) -> bool {
                const int s = t & 1;
                if (!bwait(full + s, (uint32_t)((t >> 1) & 1), p.wait_ns)) return false;
                if (t >= 2 && !bwait(s_empty + s, (uint32_t)(((t >> 1) - 1) & 1), p.wait_ns)) return false;
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(sbase + s * kSlotB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16(tmem + kColS0 + s * 64, qdesc + (uint64_t)(kk * 2), udesc + (uint64_t)(kk * 2), idS,
                              kk > 0 ? 1u : 0u);
                umma_commit(s_full + s);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int t = 0; t < T && ok; ++t) {
                const int s = t & 1;
                const uint32_t ph = (uint32_t)(t & 1);
                if (t + 1 < T && !issue_s(t + 1)) { ok = false; break; }
                // C_t = L A_t
                if (!bwait(a_full, ph, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + kColC, ldesc + (uint64_t)((((kt >> 2) * kT * 128) + (kt & 3) * 32) >> 4),
                              amn + (uint64_t)(kt * 128), idC, kt > 0 ? 1u : 0u);
                umma_commit(c_full);
                // P_t = B_t A_t^T and H_t = B_t W_pre
                if (!bwait(b_full, ph, p.wait_ns)) { ok = false; break; }
                if (t >= 1 && !(bwait(h_empty, ph ^ 1u, p.wait_ns) && bwait(wi_full, ph ^ 1u, p.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kMP / 16; ++kk)
                    umma_bf16(tmem + kColP, bk + (uint64_t)(kk * 2), ak + (uint64_t)(kk * 2), idP, kk > 0 ? 1u : 0u);
                umma_commit(p_full);
                if (t >= 1) {
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16(tmem + kColH, bk + (uint64_t)(kj * 2), wim + (uint64_t)(kj * 128), idH,
                                  kj > 0 ? 1u : 0u);
                }
                // H_t += P_t V_t, then W_pre += A_t^T V_t
                if (!bwait(pm_full, ph, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t va = sbase + s * kSlotB + kTileB;
                const uint64_t vmn = smem_desc_sw128(va, kTileB, 1024);
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + kColH, pk + (uint64_t)((((kt >> 2) * kT * 128) + (kt & 3) * 32) >> 4),
                              vmn + (uint64_t)(kt * 128), idH, (t > 0 || kt > 0) ? 1u : 0u);
                umma_commit(h_full);
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + kColW, amn + (uint64_t)(kt * 128), vmn + (uint64_t)(kt * 128), idW,
                              (t > 0 || kt > 0) ? 1u : 0u);
                umma_commit(w_full);
                umma_commit(empty + s);
            }
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        const int row = warp * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
        float a[64];
        // H of tile u out of tensor memory to global (rows past the slice are not stored)
        auto store_h = [&](int u) -> bool {
            if (!bwait(h_full, (uint32_t)(u & 1), p.wait_ns)) return false;
            tc_fence_after();
            float o[64];
            tmem_ld32(trow + kColH, o);
            tmem_ld32(trow + kColH + 32, o + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(h_empty);
            if (u * kT + row < p.n) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.H + ((size_t)slice * p.n + (size_t)(u * kT + row)) * kD);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) dst[c8] = pack8(o + 8 * c8);
            }
            return true;
        };
        for (int t = 0; t < T && ok; ++t) {
            const int s = t & 1;
            const uint32_t ph = (uint32_t)(t & 1);
            const bool valid = t * kT + row < p.n;
            // A_t (fp32, in registers)
            if (!bwait(s_full + s, (uint32_t)((t >> 1) & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColS0 + s * 64, a);
            tmem_ld32(trow + kColS0 + s * 64 + 32, a + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty + s);
            {
                const float z = rowops::softmax64_unnormalised(a, p.m, p.c);
                rowops::scale64(a, valid ? 1.f / z : 0.f);
            }
            // the tile before has finished with A, B, P and has added itself to W_pre
            if (t >= 1) {
                if (!bwait(w_full, ph ^ 1u, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
            }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + kOffA + sw_off(row, c8, kT)) = pack8(a + 8 * c8);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
            // while C_t runs: the tile before's H out, and the W_pre image for this tile (anchor
            // rows, warps 0 and 1)
            if (t >= 1) {
                if (!store_h(t - 1)) { ok = false; break; }
                if (warp < 2) {
                    float w[64];
                    tmem_ld32(trow + kColW, w);
                    tmem_ld32(trow + kColW + 32, w + 32);
                    tmem_ld_wait();
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8)
                        *reinterpret_cast<uint4 *>(sm + kOffWI + sw_off(row, c8, kMP)) = pack8(w + 8 * c8);
                    fence_proxy_async_smem();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(wi_full);
            }
            // Delta^(i) = Delta_pre + C_t[i]; B = A / Delta^(i)
            if (!bwait(c_full, ph, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            {
                float cr[64];
                tmem_ld32(trow + kColC, cr);
                tmem_ld32(trow + kColC + 32, cr + 32);
                tmem_ld_wait();
                const float *dp = sDP + s * 64;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    cr[j] = __fadd_rn(dp[j], cr[j]);
                    a[j] = cr[j] != 0.f ? __fdividef(a[j], cr[j]) : 0.f;  // rounded to bf16 next
                }
                if (row == kT - 1)  // the whole tile: the next tile's Delta_pre
#pragma unroll
                    for (int j = 0; j < 64; ++j) sDP[(s ^ 1) * 64 + j] = cr[j];
            }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + kOffB + sw_off(row, c8, kT)) = pack8(a + 8 * c8);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(b_full);
                mbar_arrive(dp_full);
            }
            // every row warp has read this tile's Delta_pre, and the next tile's is written
            if (!bwait(dp_full, ph, p.wait_ns)) { ok = false; break; }
            // P_t masked to j <= i, as the bf16 A operand of P V
            if (!bwait(p_full, ph, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float pr[64];
                tmem_ld32(trow + kColP + half * 64, pr);
                tmem_ld32(trow + kColP + half * 64 + 32, pr + 32);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (half * 64 + j > row) pr[j] = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm + kOffP + sw_off(row, half * 8 + c8, kT)) = pack8(pr + 8 * c8);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pm_full);
        }
        if (ok && T > 0) store_h(T - 1);  // the last tile's H
        __syncwarp();
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool causal_tc_supported(const Problem &p) { return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1; }

cudaError_t launch_causal_tc(const Problem &p, cudaStream_t stream) {
    CUtensorMap tq, tv, tu;
    const long long S = p.slices();
    if (!make_bf16_map(&tq, p.Q, kD, p.n, S, kT) || !make_bf16_map(&tv, p.V, kD, p.n, S, kT) ||
        !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(anchor_causal_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    CtcParams cp;
    cp.heads = p.heads;
    cp.n = p.n;
    cp.m = p.m;
    cp.tiles = (p.n + kT - 1) / kT;
    cp.c = p.scale * 1.4426950408889634f;
    cp.H = static_cast<__nv_bfloat16 *>(p.H);
    cp.wait_ns = 2000000000ull;
    return launch_pdl(anchor_causal_tc_kernel, dim3((unsigned)S), dim3(kThreads), kSmem, stream, tq, tv, tu, cp);
}

cudaError_t causal_tc_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_causal_tc_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_causal_tc_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

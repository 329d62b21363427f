// Backward of the anchor-attention forward on the tensor cores (bf16 operands, fp32
// accumulators in tensor memory) for d = 64 and m <= 64, any n.  For an upstream gradient dH
// of H = A Delta^{-1} (A^T V), A = rowsoftmax(scale Q U^T):
//   dW' = A^T dH,  dW = Delta^{-1} dW',  dDelta_j = -sum_k dW_jk W'_jk,
//   G = dH W'^T + V dW^T + 1 dDelta^T,  dS = A o (G - rowsum(A o G)),
//   dQ = scale dS U,  dV = A dW,  dU = scale dS^T Q summed over the batch entries of a head
// (the anchors are fitted by gradient descent: pith.science verdict on arXiv 2505.16463,
// "core_discovery"; the arXiv abstract, where the anchors are weights of a trainable layer).
//
// One CTA per (batch, head) slice; the slice's 128-token tiles stream twice through a
// two-slot TMA ring of [Q | V | dH] tiles:
//   B1  S_t = Q_t U^T and A_t = softmax, then W += A_t^T V_t and [dW' | Delta] += A_t^T [dH_t | 1]
//   E1  W' = W / Delta, dW = dW' / Delta and dDelta (fp32)
//   B2  S_t again and G_t = dH_t W'^T + V_t dW^T, then on CUDA cores A_t and dS_t (fp32), then
//       dQ_t = dS_t U, dV_t = A_t dW, dU += dS_t^T Q_t; dQ_t and dV_t go to global memory with
//       16-byte stores from the row that holds them
//   dU of the slice goes to a workspace row block; a second launch sums the batch entries of
//   each head in a fixed order.
// The fp32 operands that the gradients sum over many terms - A in B1, W' and dW in G, dS in dQ
// and dU - enter the MMAs as two bf16 parts, hi = bf16(x) and lo = bf16(x - hi), so they carry
// about 16 bits of mantissa: dU sums dS Q over every token of every batch entry, and a single
// bf16 rounding of each operand (8 bits) puts its error at about 1 % of dU's rms.  (A in dV,
// which sums over the m anchors only, and Q, V, dH, U, which are bf16 already, enter once.)
// Warps: 0-3 row warps (TMEM lanes 32w..32w+31: tokens, or anchors in E1 and for dU),
// 4 producer (TMA), 5 MMA issuer.  Every sum is taken in a fixed order, so the results are
// bit-identical from run to run.  Every wait is bounded; one that gives up sets bit 0 of the
// backward's error word and the CTA drains what it has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_bwd_tc_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128, kD = 64, kMP = 64;
constexpr int kThreads = 192;
constexpr int kWarpProducer = 4, kWarpMma = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileB = kT * 64 * 2;     // a 128 x 64 bf16 tile (16 KB)
constexpr int kSlotB = 3 * kTileB;      // Q | V | dH of one tile
constexpr int kImgB = kMP * kD * 2;     // a [64][64] bf16 image (8 KB)
// shared memory (an MN-major M = 128 operand reads its unused second 64-row block 16 KB on,
// so each of A_hi, A_lo, dS_hi, dS_lo has 16 KB of shared memory behind it)
constexpr int kOffAH = 2 * kSlotB;                // A_t, hi part
constexpr int kOffAL = kOffAH + kTileB;           // A_t, lo part
constexpr int kOffDSH = kOffAL + kTileB;          // dS_t, hi part
constexpr int kOffDSL = kOffDSH + kTileB;         // dS_t, lo part
constexpr int kOffImg = kOffDSL + kTileB;         // W' hi | W' lo | dW hi | dW lo images [64][64]
constexpr int kOffU = kOffImg + 4 * kImgB;        // U [64][64]
constexpr int kOffOnes = kOffU + kImgB;           // [128 tokens][64] bf16 ones
constexpr int kOffDD = kOffOnes + kTileB;         // dDelta [64] fp32
constexpr int kOffBar = kOffDD + 256;
constexpr int kBars = 24;
constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
// tensor memory columns
constexpr uint32_t kColS0 = 0;                                  // S buffers at 0 and 64 (both passes)
constexpr uint32_t kColW = 128, kColDWp = 256, kColDelta = 320; // B1 (dW' | Delta: one N = 80 result)
constexpr uint32_t kColG = 128, kColDU = 192, kColDQ0 = 256;    // B2: dQ_b, dV_b at 256 + 128 b

struct BtcParams {
    int heads, n, m, tiles;
    float c;        // scale * log2(e)
    float scale;
    float *dupart;  // [slices][m][64]
    __nv_bfloat16 *dQ, *dV;
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
// bf16 parts of 8 floats: hi = round(x), lo = round(x - hi)
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = x[i] - __bfloat162float(__float2bfloat16_rn(x[i]));
    hi = pack8(x, 1.f);
    lo = pack8(r, 1.f);
}

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_bwd_tc_error, 1u);
            return false;
        }
    }
    return true;
}

// row softmax of 64 scores (anchors >= m masked), in place; a row past the slice is all zero
__device__ __forceinline__ void softmax64(float (&v)[64], int m, float c, bool valid) {
    const float z = rowops::softmax64_unnormalised(v, m, c);
    rowops::scale64(v, valid ? 1.f / z : 0.f);
}

// a row of 64 fp32 values as hi and lo bf16 rows of a swizzled [rows][64] tile
__device__ __forceinline__ void store_split(uint8_t *hi, uint8_t *lo, int row, int rows, const float *x) {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 h, l;
        split8(x + 8 * c8, h, l);
        *reinterpret_cast<uint4 *>(hi + sw_off(row, c8, rows)) = h;
        *reinterpret_cast<uint4 *>(lo + sw_off(row, c8, rows)) = l;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
anchor_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ CUtensorMap tdh, const __grid_constant__ CUtensorMap tu,
                     const BtcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *full = bars + 0, *empty = bars + 2, *u_full = bars + 4;
    uint64_t *s_full = bars + 5, *s_empty = bars + 7, *a_full = bars + 9, *a_empty = bars + 10;
    uint64_t *w_full = bars + 11, *ep_full = bars + 12, *g_full = bars + 13, *g_empty = bars + 14;
    uint64_t *ds_full = bars + 15, *ds_empty = bars + 16, *dqv_full = bars + 17, *dqv_empty = bars + 19;
    uint64_t *du_full = bars + 21, *mma_done = bars + 22;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);
    float *sDD = reinterpret_cast<float *>(sm + kOffDD);

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
            mbar_init(dqv_full + i, 1);
            mbar_init(dqv_empty + i, 4);
        }
        mbar_init(u_full, 1);
        mbar_init(a_full, 4);
        mbar_init(a_empty, 1);
        mbar_init(w_full, 1);
        mbar_init(ep_full, 4);
        mbar_init(g_full, 1);
        mbar_init(g_empty, 4);
        mbar_init(ds_full, 4);
        mbar_init(ds_empty, 1);
        mbar_init(du_full, 1);
        mbar_init(mma_done, 1);
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
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdh);
            tma_prefetch_desc(&tu);
            const uint64_t pol_keep = policy_evict_last(), pol_once = policy_evict_first();
            mbar_arrive_expect_tx(u_full, kImgB);
            tma_load_3d(sm + kOffU, &tu, u_full, 0, 0, h, pol_keep);
            int issued = 0;
            for (int seq = 0; seq < 2 * T; ++seq) {
                const int s = seq & 1, t = seq < T ? seq : seq - T;
                if (seq >= 2 && !bwait(empty + s, (uint32_t)(((seq >> 1) - 1) & 1), p.wait_ns)) break;
                uint8_t *st = sm + s * kSlotB;
                // the second pass is the tile's last read: evict-first then
                const uint64_t pol = seq < T ? pol_keep : pol_once;
                mbar_arrive_expect_tx(full + s, 3 * kTileB);
                tma_load_3d(st, &tq, full + s, 0, t * kT, slice, pol);
                tma_load_3d(st + kTileB, &tv, full + s, 0, t * kT, slice, pol);
                tma_load_3d(st + 2 * kTileB, &tdh, full + s, 0, t * kT, slice, pol);
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
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);    // [tokens x anchors], K = d
            const uint32_t idW = idesc_bf16_f32(kT, kD, true, true);       // A^T X: anchors x d, K = tokens
            const uint32_t idWD = idesc_bf16_f32(kT, kD + 16, true, true); // A^T [dH | 1]
            const uint32_t idR = idesc_bf16_f32(kT, kD, false, true);      // [tokens x d], K = anchors
            const uint64_t udesc = smem_desc_sw128(sbase + kOffU, 16, 1024);         // U, K-major
            const uint64_t umn = smem_desc_sw128(sbase + kOffU, kMP * 128, 1024);    // U, MN-major
            const uint32_t img = sbase + kOffImg;
            bool ok = bwait(u_full, 0u, p.wait_ns);
            // S_u (u: global S index, B1 tiles then B2 tiles) of the tile in ring slot (u & 1)
            auto issue_s = [&](int u) -> bool {
                const int s = u & 1, b = u & 1;
                if (!bwait(full + s, (uint32_t)((u >> 1) & 1), p.wait_ns)) return false;
                if (u >= 2 && !bwait(s_empty + b, (uint32_t)(((u >> 1) - 1) & 1), p.wait_ns)) return false;
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(sbase + s * kSlotB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16(tmem + kColS0 + b * 64, qdesc + (uint64_t)(kk * 2), udesc + (uint64_t)(kk * 2), idS,
                              kk > 0 ? 1u : 0u);
                umma_commit(s_full + b);
                return true;
            };
            // ------------------------------------------------------------------ B1
            if (ok) ok = issue_s(0);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T && !issue_s(t + 1)) { ok = false; break; }
                const int s = t & 1;
                if (!bwait(a_full, (uint32_t)(t & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sl = sbase + s * kSlotB;
                const uint64_t vdesc = smem_desc_sw128(sl + kTileB, kTileB, 1024);
                // [dH | 1]: the ones block is the operand's second 64-column block
                const uint64_t hdesc = smem_desc_sw128(sl + 2 * kTileB, (sbase + kOffOnes) - (sl + 2 * kTileB), 1024);
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint64_t adesc = smem_desc_sw128(sbase + (part ? kOffAL : kOffAH), kTileB, 1024);
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt) {
                        const uint32_t acc = (t > 0 || part > 0 || kt > 0) ? 1u : 0u;
                        const uint64_t ak = adesc + (uint64_t)(kt * 128);
                        umma_bf16(tmem + kColW, ak, vdesc + (uint64_t)(kt * 128), idW, acc);
                        umma_bf16(tmem + kColDWp, ak, hdesc + (uint64_t)(kt * 128), idWD, acc);
                    }
                }
                umma_commit(a_empty);
                umma_commit(empty + s);
            }
            if (ok) umma_commit(w_full);
            // ------------------------------------------------------------------ B2
            // G_t = dH_t (W'_hi + W'_lo)^T + V_t (dW_hi + dW_lo)^T (tile t in ring slot s)
            auto issue_g = [&](int t) -> bool {
                const int s = (T + t) & 1;
                if (t >= 1 && !bwait(g_empty, (uint32_t)((t - 1) & 1), p.wait_ns)) return false;
                tc_fence_after();
                const uint32_t sl = sbase + s * kSlotB;
                const uint64_t vk = smem_desc_sw128(sl + kTileB, 16, 1024);
                const uint64_t hk = smem_desc_sw128(sl + 2 * kTileB, 16, 1024);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t ad = i < 2 ? hk : vk;
                    const uint64_t bd = smem_desc_sw128(img + i * kImgB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        umma_bf16(tmem + kColG, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idS,
                                  (i > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(g_full);
                return true;
            };
            // S and G of the next tile are issued before this tile's dQ, dV and dU, so that the
            // row warps find them ready when they finish this tile
            if (ok) ok = issue_s(T);
            ok = ok && bwait(ep_full, 0u, p.wait_ns) && issue_g(0);
            for (int t = 0; t < T && ok; ++t) {
                const int u = T + t, s = u & 1, b = t & 1;
                if (t + 1 < T && !(issue_s(u + 1) && issue_g(t + 1))) { ok = false; break; }
                const uint32_t sl = sbase + s * kSlotB;
                // dQ_t, dV_t and dU once the row warps have written dS_t and A_t
                if (!bwait(ds_full, (uint32_t)(t & 1), p.wait_ns)) { ok = false; break; }
                if (t >= 2 && !bwait(dqv_empty + b, (uint32_t)(((t >> 1) - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t cq = kColDQ0 + b * 128;
                const uint64_t ak = smem_desc_sw128(sbase + kOffAH, 16, 1024);
#pragma unroll
                for (int i = 0; i < 2; ++i) {  // dV = A (dW_hi + dW_lo)
                    const uint64_t dwm = smem_desc_sw128(img + (2 + i) * kImgB, kMP * 128, 1024);
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16(tmem + cq + 64, ak + (uint64_t)(kj * 2), dwm + (uint64_t)(kj * 128), idR,
                                  (i > 0 || kj > 0) ? 1u : 0u);
                }
                const uint64_t qm = smem_desc_sw128(sl, kTileB, 1024);     // Q_t, MN-major (N = d)
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint32_t da = sbase + (part ? kOffDSL : kOffDSH);
                    const uint64_t dsk = smem_desc_sw128(da, 16, 1024);
                    const uint64_t dsm = smem_desc_sw128(da, kTileB, 1024);   // dS^T: anchors x tokens
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16(tmem + cq, dsk + (uint64_t)(kj * 2), umn + (uint64_t)(kj * 128), idR,
                                  (part > 0 || kj > 0) ? 1u : 0u);
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt)
                        umma_bf16(tmem + kColDU, dsm + (uint64_t)(kt * 128), qm + (uint64_t)(kt * 128), idW,
                                  (t > 0 || part > 0 || kt > 0) ? 1u : 0u);
                }
                umma_commit(dqv_full + b);
                umma_commit(ds_empty);
                umma_commit(empty + s);
            }
            if (ok) umma_commit(du_full);
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        const int row = warp * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        {   // the ones block (every element 1; the MMA reads columns 0..15 of each token row)
            const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
            for (int i = row; i < kTileB / 16; i += 128) reinterpret_cast<uint4 *>(sm + kOffOnes)[i] = ones;
        }
        bool ok = true;
        float v[64];
        // B1: A_t of every tile
        for (int t = 0; t < T && ok; ++t) {
            const int b = t & 1;
            if (!bwait(s_full + b, (uint32_t)((t >> 1) & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColS0 + b * 64, v);
            tmem_ld32(trow + kColS0 + b * 64 + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty + b);
            softmax64(v, p.m, p.c, t * kT + row < p.n);
            if (t >= 1 && !bwait(a_empty, (uint32_t)((t - 1) & 1), p.wait_ns)) { ok = false; break; }
            store_split(sm + kOffAH, sm + kOffAL, row, kT, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
        }
        // E1: anchor j = row (warps 0, 1)
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
                for (int k = 0; k < 64; ++k) w[k] *= rinv;  // W'
                store_split(sm + kOffImg, sm + kOffImg + kImgB, row, kMP, w);
                tmem_ld32(trow + kColDWp, v);
                tmem_ld32(trow + kColDWp + 32, v + 32);
                tmem_ld_wait();
                float dd = 0.f;
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    v[k] *= rinv;  // dW
                    dd = fmaf(v[k], w[k], dd);
                }
                store_split(sm + kOffImg + 2 * kImgB, sm + kOffImg + 3 * kImgB, row, kMP, v);
                sDD[row] = dl[0] != 0.f ? -dd : 0.f;
                fence_proxy_async_smem();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ep_full);
        }
        ok = ok && bwait(ep_full, 0u, p.wait_ns);
        // B2: dS_t and A_t, then the stores of dQ and dV of the tile before
        auto drain = [&](int t) -> bool {
            const int b = t & 1;
            if (!bwait(dqv_full + b, (uint32_t)((t >> 1) & 1), p.wait_ns)) return false;
            tc_fence_after();
            float o[64];
            const bool valid = t * kT + row < p.n;
            const size_t off = ((size_t)slice * p.n + (size_t)(t * kT + row)) * kD;
            tmem_ld32(trow + kColDQ0 + b * 128, o);
            tmem_ld32(trow + kColDQ0 + b * 128 + 32, o + 32);
            tmem_ld_wait();
            if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.dQ + off);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) dst[c8] = pack8(o + 8 * c8, p.scale);
            }
            tmem_ld32(trow + kColDQ0 + b * 128 + 64, o);
            tmem_ld32(trow + kColDQ0 + b * 128 + 96, o + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dqv_empty + b);
            if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.dV + off);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) dst[c8] = pack8(o + 8 * c8, 1.f);
            }
            return true;
        };
        for (int t = 0; t < T && ok; ++t) {
            const int u = T + t, bs = u & 1;
            if (!bwait(s_full + bs, (uint32_t)((u >> 1) & 1), p.wait_ns)) { ok = false; break; }
            if (!bwait(g_full, (uint32_t)(t & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            float g[64];
            tmem_ld32(trow + kColS0 + bs * 64, v);
            tmem_ld32(trow + kColS0 + bs * 64 + 32, v + 32);
            tmem_ld32(trow + kColG, g);
            tmem_ld32(trow + kColG + 32, g + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(s_empty + bs);
                mbar_arrive(g_empty);
            }
            softmax64(v, p.m, p.c, t * kT + row < p.n);
            // dS_j = A_j (G_j + dDelta_j - sum_l A_l (G_l + dDelta_l))
#pragma unroll
            for (int j = 0; j < 64; ++j) g[j] += sDD[j];
            const float rs = rowops::dot64(v, g);
#pragma unroll
            for (int j = 0; j < 64; ++j) g[j] = v[j] * (g[j] - rs);
            if (t >= 1 && !bwait(ds_empty, (uint32_t)((t - 1) & 1), p.wait_ns)) { ok = false; break; }
            store_split(sm + kOffDSH, sm + kOffDSL, row, kT, g);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + kOffAH + sw_off(row, c8, kT)) = pack8(v + 8 * c8, 1.f);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
            if (t >= 1 && !drain(t - 1)) { ok = false; break; }
        }
        if (ok && T >= 1) ok = drain(T - 1);
        // dU of this slice (scale dS^T Q): anchor j = row, warps 0 and 1
        ok = ok && bwait(du_full, 0u, p.wait_ns);
        if (ok && warp < 2) {
            tc_fence_after();
            tmem_ld32(trow + kColDU, v);
            tmem_ld32(trow + kColDU + 32, v + 32);
            tmem_ld_wait();
            if (row < p.m) {
                float4 *dst = reinterpret_cast<float4 *>(p.dupart + ((size_t)slice * p.m + row) * kD);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    dst[k] = make_float4(v[4 * k] * p.scale, v[4 * k + 1] * p.scale, v[4 * k + 2] * p.scale,
                                         v[4 * k + 3] * p.scale);
            }
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

bool bwd_tc_supported(const BwdProblem &p) { return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1; }

size_t bwd_tc_workspace(const BwdProblem &p) { return (size_t)p.slices() * p.m * kD * 4; }

cudaError_t launch_bwd_tc(const BwdProblem &p, void *workspace, cudaStream_t stream) {
    CUtensorMap tq, tv, tdh, tu;
    const long long S = p.slices();
    if (!make_bf16_map(&tq, p.Q, kD, p.n, S, kT) || !make_bf16_map(&tv, p.V, kD, p.n, S, kT) ||
        !make_bf16_map(&tdh, p.dH, kD, p.n, S, kT) || !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(anchor_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    BtcParams bp;
    bp.heads = p.heads;
    bp.n = p.n;
    bp.m = p.m;
    bp.tiles = (p.n + kT - 1) / kT;
    bp.c = p.scale * 1.4426950408889634f;
    bp.scale = p.scale;
    bp.dupart = static_cast<float *>(workspace);
    bp.dQ = static_cast<__nv_bfloat16 *>(p.dQ);
    bp.dV = static_cast<__nv_bfloat16 *>(p.dV);
    bp.wait_ns = 2000000000ull;
    if ((e = launch_pdl(anchor_bwd_tc_kernel, dim3((unsigned)S), dim3(kThreads), kSmem, stream, tq, tv, tdh, tu, bp)) !=
        cudaSuccess)
        return e;
    return launch_bwd_du_sum(bp.dupart, p.dU, p.B, p.heads, 1, p.m * kD, false, stream);
}

cudaError_t bwd_tc_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_tc_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_bwd_tc_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

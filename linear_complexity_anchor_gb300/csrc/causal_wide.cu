// Masked (causal) variant of the anchor-attention forward on the tensor cores for up to 128
// anchors (bf16 operands, fp32 accumulators in tensor memory), d = 64 or 128, any n.  Token
// i's anchor summaries include only tokens j <= i (one of the inferences of the pith.science
// verdict on arXiv 2505.16463: A can be masked against later tokens without giving up the
// O(mn) cost):
//   Delta^(i)_l = sum_{j<=i} A[j][l],  W^(i)_l = sum_{j<=i} A[j][l] v_j,
//   H[i] = sum_l A[i][l] W^(i)_l / Delta^(i)_l   (0 for an anchor with Delta^(i)_l = 0).
//
// The same tile recurrence as the kernel for 64 anchors (causal_tc.cu), laid out for 128-wide
// anchor rows: one CTA per (batch, head) slice walks the slice's 128-token tiles in order,
// keeping the summaries of the tiles before (W_pre in tensor memory, Delta_pre in shared
// memory).  Per tile t, with B[i][l] = A[i][l] / Delta^(i)_l:
//   S_t = Q_t U^T, A_t = softmax (row warps)
//   C_t = L A_t (L the lower-triangular ones: running column sums inside the tile), so
//         Delta^(i) = Delta_pre + C_t[i]; the row warps form B_t
//   P_t = B_t A_t^T, masked to j <= i by the row warps
//   H_t = B_t W_pre + P_t V_t
//   W_pre += A_t^T V_t, Delta_pre += the tile's column sums (the last row of C_t)
// The sums over j use the bf16 A_t in every place (C_t, P_t, W_pre), so Delta and W stay
// consistent; B on the i side is formed from the fp32 A.
//
// What differs from the 64-anchor layout, so that it fits 227 KB of shared memory and 512
// tensor-memory columns at d = m = 128: Q_t and V_t have one buffer each (Q_{t+1} loads once
// S_t has read Q_t, V_{t+1} once the tile's last MMA has read V_t, both well before they are
// needed); C_t goes into S_t's columns (the row warps have read S_t by then); the masked P_t
// goes over B_t (every MMA reading B_t has completed by then).  Shared memory (D = 128): Q, V,
// U, L, A, B / P, W_pre image, 32 KB each.  Tensor memory: S / C at 0, P at 128, H at 256,
// W_pre at 384.
// Warps: 0-7 row warps (warp w: TMEM lanes 32 (w % 4) .. + 31, tokens or anchors for the
// W_pre image; half w / 4 of the columns, the softmax's (max, sum) pairs exchanged through
// tensor memory; a tile's H goes out while the next tile's C runs, staged in the warp's own
// rows of the B / P tile and written by TMA stores), 8 producer (TMA), 9 MMA issuer.  Sums run
// in a fixed order: results are bit-identical from run to run.  Every wait is bounded; one
// that gives up sets bit 0 of this kernel's error word and the CTA drains what it has in
// flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"
#include "tmem_pair.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_causal_wide_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128, kMP = 128;
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;  // warps 0-7: row warps
constexpr uint32_t kTmemCols = 512;
constexpr int kBlkB = kT * 64 * 2;  // a [128][64] bf16 block (16 KB)
constexpr uint32_t kColSC = 0, kColP = 128, kColH = 256, kColW = 384;

template <int D>
struct WideLayout {
    static constexpr int kQB = D / 64 * kBlkB;   // [128][D]
    static constexpr int kOffQ = 0;
    static constexpr int kOffV = kOffQ + kQB;
    static constexpr int kOffU = kOffV + kQB;     // [128 anchors][D]
    static constexpr int kOffL = kOffU + kQB;     // [128][128]
    static constexpr int kOffA = kOffL + 2 * kBlkB;
    static constexpr int kOffB = kOffA + 2 * kBlkB;   // B_t, then the masked P_t
    static constexpr int kOffWI = kOffB + 2 * kBlkB;  // W_pre image [128 anchors][D]
    static constexpr int kOffDP = kOffWI + kQB;       // Delta_pre [2][128] fp32
    static constexpr int kOffBar = kOffDP + 1024;
    static constexpr int kBars = 24;
    static constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(kColW + D <= kTmemCols && kColH + D <= kColW, "tensor memory columns");
};

struct CwParams {
    int heads, n, m, tiles;
    int chunks;  // CTAs per slice (token chunks); chunk c first sums the tiles before it
    float c;  // scale * log2(e)
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
// K-step kk of a K-major operand of `rows` rows stored as 64-column blocks
__device__ __forceinline__ uint64_t kstep(int kk, int rows) {
    return (uint64_t)((((kk >> 2) * rows * 128) + (kk & 3) * 32) >> 4);
}

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_causal_wide_error, 1u);
            return false;
        }
    }
    return true;
}

// First tile of chunk c of a slice's `tiles` tiles.  A chunk first walks the tiles before it
// as summary tiles (S, A and the summaries' products only), which cost about kSummaryCost of a
// full tile, so later chunks get fewer full tiles: the boundaries equalise
// (full tiles) + kSummaryCost * (summary tiles) over the chunks.
constexpr float kSummaryCost = 0.5f;
__host__ __device__ __forceinline__ int chunk_bound(int c, int tiles, int chunks) {
    if (c <= 0) return 0;
    if (c >= chunks) return tiles;
    if (kSummaryCost <= 0.f) return (int)((long long)c * tiles / chunks);
    const float r = 1.f - kSummaryCost;
    float rc = 1.f, rk = 1.f;
    for (int i = 0; i < c; ++i) rc *= r;
    for (int i = 0; i < chunks; ++i) rk *= r;
    const int b = (int)((float)tiles * (1.f - rc) / (1.f - rk) + 0.5f);
    return b < c ? c : (b > tiles - (chunks - c) ? tiles - (chunks - c) : b);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
anchor_causal_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap th,
                          const CwParams p) {
    using LY = WideLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::kOffBar);
    uint64_t *q_full = bars + 0, *q_empty = bars + 1, *v_full = bars + 2, *v_empty = bars + 3;
    uint64_t *u_full = bars + 4, *s_full = bars + 5, *a_full = bars + 6, *c_full = bars + 7, *b_full = bars + 8;
    uint64_t *p_full = bars + 9, *pm_full = bars + 10, *h_full = bars + 11, *h_empty = bars + 12;
    uint64_t *w_full = bars + 13, *wi_full = bars + 14, *mma_done = bars + 15, *dp_full = bars + 16;
    uint64_t *x_sm = bars + 17;  // the two halves' (max, sum) pairs written
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + LY::kBars);
    float *sDP = reinterpret_cast<float *>(sm + LY::kOffDP);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x / p.chunks, chunk = blockIdx.x - slice * p.chunks;
    const int h = slice % p.heads;
    // this CTA's tiles: [t0, t1) of the slice; tiles [0, t0) run first as summary tiles (S,
    // softmax, C for Delta, W only), which leave W_pre and Delta_pre exactly as a CTA that
    // ran them in full would (the same MMAs and additions in the same order)
    const int t0 = chunk_bound(chunk, p.tiles, p.chunks), t1 = chunk_bound(chunk + 1, p.tiles, p.chunks);
    const int T = t1;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(u_full, 1);
        mbar_init(s_full, 1);
        mbar_init(a_full, 8);
        mbar_init(c_full, 1);
        mbar_init(b_full, 8);
        mbar_init(p_full, 1);
        mbar_init(pm_full, 8);
        mbar_init(h_full, 1);
        mbar_init(h_empty, 8);
        mbar_init(w_full, 1);
        mbar_init(wi_full, 8);
        mbar_init(mma_done, 1);
        mbar_init(dp_full, 8);
        mbar_init(x_sm, 8);
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
            *reinterpret_cast<uint4 *>(sm + LY::kOffL + sw_off(row, c8, kT)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        sDP[row] = 0.f;
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
            tma_prefetch_desc(&th);
            const uint64_t pol_keep = policy_evict_last(), pol_once = policy_evict_first();
            mbar_arrive_expect_tx(u_full, LY::kQB);
#pragma unroll
            for (int b = 0; b < D / 64; ++b) tma_load_3d(sm + LY::kOffU + b * kBlkB, &tu, u_full, 64 * b, 0, h, pol_keep);
            int nq = 0, nv = 0;
            bool ok = true;
            for (int t = 0; t < T && ok; ++t) {
                // Q_t once S_{t-1} has read Q_{t-1}; V_t once the MMAs of tile t-1 have read V_{t-1}
                if (t >= 1 && !bwait(q_empty, (uint32_t)((t - 1) & 1), p.wait_ns)) { ok = false; break; }
                mbar_arrive_expect_tx(q_full, LY::kQB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sm + LY::kOffQ + b * kBlkB, &tq, q_full, 64 * b, t * kT, slice, pol_once);
                ++nq;
                if (t >= 1 && !bwait(v_empty, (uint32_t)((t - 1) & 1), p.wait_ns)) { ok = false; break; }
                mbar_arrive_expect_tx(v_full, LY::kQB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sm + LY::kOffV + b * kBlkB, &tv, v_full, 64 * b, t * kT, slice, pol_once);
                ++nv;
            }
            // leave no copy in flight
            if (nq > 0) bwait(q_full, (uint32_t)((nq - 1) & 1), p.wait_ns);
            if (nv > 0) bwait(v_full, (uint32_t)((nv - 1) & 1), p.wait_ns);
            bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);   // Q U^T: [tokens x anchors], K = d
            const uint32_t idC = idesc_bf16_f32(kT, kMP, false, true);    // L A: K = tokens
            const uint32_t idP = idesc_bf16_f32(kT, kT, false, false);    // B A^T: [tokens x tokens], K = anchors
            const uint32_t idH = idesc_bf16_f32(kT, D, false, true);      // [tokens x d]
            const uint32_t idW = idesc_bf16_f32(kMP, D, true, true);      // A^T V: anchors x d, K = tokens
            const uint64_t qdesc = smem_desc_sw128(sbase + LY::kOffQ, 16, 1024);
            const uint64_t udesc = smem_desc_sw128(sbase + LY::kOffU, 16, 1024);
            const uint64_t ldesc = smem_desc_sw128(sbase + LY::kOffL, 16, 1024);
            const uint64_t amn = smem_desc_sw128(sbase + LY::kOffA, kBlkB, 1024);   // A_t, MN-major
            const uint64_t ak = smem_desc_sw128(sbase + LY::kOffA, 16, 1024);       // A_t, K-major
            const uint64_t bk = smem_desc_sw128(sbase + LY::kOffB, 16, 1024);       // B_t / P_t, K-major
            const uint64_t vmn = smem_desc_sw128(sbase + LY::kOffV, kBlkB, 1024);   // V_t, MN-major
            const uint64_t wim = smem_desc_sw128(sbase + LY::kOffWI, kBlkB, 1024);  // W_pre image, MN-major
            bool ok = bwait(u_full, 0u, p.wait_ns);
            auto issue_s = [&](int t) -> bool {  // S_t into the S / C columns
                if (!bwait(q_full, (uint32_t)(t & 1), p.wait_ns)) return false;
                // C_{t-1} read (a full tile's C shares S's columns; a summary tile's is in P's)
                if (t - 1 >= t0 && !bwait(b_full, (uint32_t)((t - 1) & 1), p.wait_ns)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_bf16(tmem + kColSC, qdesc + kstep(kk, kT), udesc + kstep(kk, kMP), idS, kk > 0 ? 1u : 0u);
                umma_commit(s_full);
                umma_commit(q_empty);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int t = 0; t < T && ok; ++t) {
                const uint32_t ph = (uint32_t)(t & 1);
                const bool full = t >= t0;
                const int u = t - t0;                         // full tile index
                const int img = u - (t0 == 0 ? 1 : 0);        // W_pre image index (full tiles with t >= 1)
                // C_t = L A_t over S_t's columns (a summary tile's over P's, so that S_{t+1} need
                // not wait for it to be read)
                if (!bwait(a_full, ph, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t ccol = full ? kColSC : kColP;
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + ccol, ldesc + kstep(kt, kT), amn + (uint64_t)(kt * 128), idC, kt > 0 ? 1u : 0u);
                umma_commit(c_full);
                if (full) {
                    // P_t = B_t A_t^T and H_t = B_t W_pre
                    if (!bwait(b_full, ph, p.wait_ns)) { ok = false; break; }
                    if (u >= 1 && !bwait(h_empty, (uint32_t)((u - 1) & 1), p.wait_ns)) { ok = false; break; }
                    if (t >= 1 && !bwait(wi_full, (uint32_t)(img & 1), p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kMP / 16; ++kk)
                        umma_bf16(tmem + kColP, bk + kstep(kk, kT), ak + kstep(kk, kT), idP, kk > 0 ? 1u : 0u);
                    if (t >= 1) {
#pragma unroll
                        for (int kj = 0; kj < kMP / 16; ++kj)
                            umma_bf16(tmem + kColH, bk + kstep(kj, kT), wim + (uint64_t)(kj * 128), idH, kj > 0 ? 1u : 0u);
                    }
                    umma_commit(p_full);
                }
                // the next tile's scores while the row warps mask P_t (or once they have read C_t)
                if (t + 1 < T && !issue_s(t + 1)) { ok = false; break; }
                if (full) {
                    // H_t += P_t V_t
                    if (!bwait(pm_full, (uint32_t)(u & 1), p.wait_ns) || !bwait(v_full, ph, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt)
                        umma_bf16(tmem + kColH, bk + kstep(kt, kT), vmn + (uint64_t)(kt * 128), idH,
                                  (t > 0 || kt > 0) ? 1u : 0u);
                    umma_commit(h_full);
                } else {
                    if (!bwait(v_full, ph, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                }
                // W_pre += A_t^T V_t
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + kColW, amn + (uint64_t)(kt * 128), vmn + (uint64_t)(kt * 128), idW,
                              (t > 0 || kt > 0) ? 1u : 0u);
                umma_commit(w_full);
                umma_commit(v_empty);
            }
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (tokens; anchors for the W_pre image), column
        // half g = w / 4 (anchors 64 g .. 64 g + 63 of S, C and B; tokens 64 g .. of P; the
        // columns D/2 g .. of H and of the W_pre image)
        const int q4 = warp & 3, g = warp >> 2;
        const int row = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        constexpr int DH = D / 2;  // this half's columns of H and of the W_pre image
        bool ok = true;
        float a[64];
        // H of full tile u (slice tile t0 + u): tensor memory -> this warp's own rows of the
        // B / P tile (free: the tile's H products have read P; the same swizzled layout as a
        // [32][64] TMA box) -> a TMA store (rows past the slice are not written).  At D = 128
        // each half stores its 64 columns; at D = 64 half 0 stores all of them.  The warp's
        // next B rows are written once its stores have read them.
        const uint64_t pol_out = policy_evict_first();
        auto store_h = [&](int u) -> bool {
            if (!bwait(h_full, (uint32_t)(u & 1), p.wait_ns)) return false;
            tc_fence_after();
            const bool mine = D == 128 || g == 0;
            if (mine) {
                const int c0 = D == 128 ? 64 * g : 0;  // this warp's 64 columns of H
                uint8_t *box = sm + LY::kOffB + g * kBlkB + q4 * 4096;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float o[32];
                    tmem_ld32(trow + kColH + c0 + q * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(box + sw_off(lane, q * 4 + c, 32)) = pack8(o + 8 * c);
                }
            }
            tc_fence_before();
            __syncwarp();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(h_empty);
                if (mine) {
                    tma_store_3d(&th, sm + LY::kOffB + g * kBlkB + q4 * 4096, D == 128 ? 64 * g : 0,
                                 (t0 + u) * kT + q4 * 32, slice, pol_out);
                    bulk_commit_group();
                }
            }
            return true;
        };
        auto stores_read = [&]() {  // this warp's H stores have read its B rows
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
        };
        for (int t = 0; t < T && ok; ++t) {
            const uint32_t ph = (uint32_t)(t & 1);
            const bool valid = t * kT + row < p.n;
            const bool full = t >= t0;
            const int u = t - t0;  // full tile index
            // A_t (fp32, in registers): this half's maximum, exponentials and sum; the halves'
            // (max, sum) pairs exchanged through the last two of each half's own S columns (C_t
            // goes there only once every row warp has passed a_full); both halves scaled to the
            // row's maximum M: A_j = e_j 2^(m_g - M) / (z_0 2^(m_0 - M) + z_1 2^(m_1 - M))
            if (!bwait(s_full, ph, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            {
                tmem_ld32(trow + kColSC + 64 * g, a);
                tmem_ld32(trow + kColSC + 64 * g + 32, a + 32);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 64; ++j) a[j] = 64 * g + j < p.m ? a[j] * p.c : -INFINITY;
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = a[k];
#pragma unroll
                for (int j = 8; j < 64; j += 8)
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], a[j + k]);
                const float mg = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float ms = mg == -INFINITY ? 0.f : mg;  // a half with every anchor masked
                float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    a[j] = rowops::ex2_approx(a[j] - ms);
                    z4[j & 3] += a[j];
                }
                const float2 mine = make_float2(mg, (z4[0] + z4[1]) + (z4[2] + z4[3]));
                tmem_st2(trow + kColSC + 64 * g + 62, mine.x, mine.y);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(x_sm);
                if (!bwait(x_sm, ph, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const float2 other = tmem_ld2(trow + kColSC + 64 * (1 - g) + 62);
                tmem_ld_wait();
                const float2 h0 = g == 0 ? mine : other, h1 = g == 0 ? other : mine;
                const float M = fmaxf(h0.x, h1.x);  // finite: half 0 holds anchor 0
                const float f0 = h0.x == -INFINITY ? 0.f : rowops::ex2_approx(h0.x - M);
                const float f1 = h1.x == -INFINITY ? 0.f : rowops::ex2_approx(h1.x - M);
                const float r = valid ? (g == 0 ? f0 : f1) / (h0.y * f0 + h1.y * f1) : 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) a[j] *= r;
            }
            // the tile before has finished with A, B, P and has added itself to W_pre
            if (t >= 1) {
                if (!bwait(w_full, ph ^ 1u, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
            }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + LY::kOffA + sw_off(row, 8 * g + c8, kT)) = pack8(a + 8 * c8);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
            if (!full) {
                // a summary tile: Delta_pre += the tile's column sums (the last row of C_t, in
                // the P columns), by the last rows' warps (tensor-memory loads are warp-wide);
                // the other warps go on to the next tile
                if (q4 == (kT - 1) / 32) {
                    if (!bwait(c_full, ph, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const float *dp = sDP + (t & 1) * kMP + 64 * g;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float cr[32];
                        tmem_ld32(trow + kColP + 64 * g + q * 32, cr);
                        tmem_ld_wait();
                        if (row == kT - 1)
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                sDP[((t + 1) & 1) * kMP + 64 * g + q * 32 + j] = __fadd_rn(dp[q * 32 + j], cr[j]);
                    }
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(b_full);
                    mbar_arrive(dp_full);
                }
                continue;
            }
            // while C_t runs: the tile before's H out, and this half of the W_pre image for
            // this tile (anchor rows)
            if (t >= 1) {
                if (u >= 1 && !store_h(u - 1)) { ok = false; break; }
#pragma unroll
                for (int q = 0; q < DH / 32; ++q) {
                    float w[32];
                    tmem_ld32(trow + kColW + DH * g + q * 32, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(sm + LY::kOffWI + sw_off(row, (DH * g) / 8 + q * 4 + c, kMP)) =
                            pack8(w + 8 * c);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(wi_full);
            }
            stores_read();
            // Delta^(i) = Delta_pre + C_t[i]; B = A / Delta^(i).  The first full tile after
            // summary tiles reads the Delta_pre the last of them wrote.
            if (u == 0 && t0 > 0 && !bwait(dp_full, (uint32_t)((t0 - 1) & 1), p.wait_ns)) { ok = false; break; }
            if (!bwait(c_full, ph, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            {
                const float *dp = sDP + (t & 1) * kMP + 64 * g;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float cr[32];
                    tmem_ld32(trow + kColSC + 64 * g + q * 32, cr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        cr[j] = __fadd_rn(dp[q * 32 + j], cr[j]);
                        a[q * 32 + j] = cr[j] != 0.f ? __fdividef(a[q * 32 + j], cr[j]) : 0.f;  // rounded to bf16 next
                    }
                    if (row == kT - 1)  // the whole tile: the next tile's Delta_pre
#pragma unroll
                        for (int j = 0; j < 32; ++j) sDP[((t + 1) & 1) * kMP + 64 * g + q * 32 + j] = cr[j];
                }
            }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sm + LY::kOffB + sw_off(row, 8 * g + c8, kT)) = pack8(a + 8 * c8);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(b_full);
                mbar_arrive(dp_full);
            }
            // every row warp has read this tile's Delta_pre, and the next tile's is written
            if (!bwait(dp_full, ph, p.wait_ns)) { ok = false; break; }
            // P_t masked to j <= i, over B_t, as the A operand of P V (this half: tokens 64 g ..)
            if (!bwait(p_full, (uint32_t)(u & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float pr[32];
                tmem_ld32(trow + kColP + 64 * g + q * 32, pr);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (64 * g + q * 32 + j > row) pr[j] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(sm + LY::kOffB + sw_off(row, 8 * g + q * 4 + c, kT)) = pack8(pr + 8 * c);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pm_full);
        }
        if (ok && t1 > t0) store_h(t1 - t0 - 1);  // the last tile's H
        if (lane == 0) bulk_wait_group0();       // the stores have landed
        __syncwarp();
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// CTAs per slice: with fewer slices than SMs, the tokens of a slice are cut into up to four
// chunks of at least four tiles, one CTA each (one CTA per SM), at the boundaries
// chunk_bound gives.  The chunk boundaries do not change the results (each chunk first sums
// the tiles before it in the same order).
int causal_wide_chunks(long long slices, int tiles) {
    long long k = kPlanSMs / (slices > 0 ? slices : 1);
    k = k < 1 ? 1 : (k > 4 ? 4 : k);
    while (k > 1 && tiles / k < 4) --k;
    return (int)k;
}

template <int D>
cudaError_t launch_d(const Problem &p, cudaStream_t stream) {
    using LY = WideLayout<D>;
    CUtensorMap tq, tv, tu, th;
    const long long S = p.slices();
    if (!make_bf16_map(&tq, p.Q, D, p.n, S, kT) || !make_bf16_map(&tv, p.V, D, p.n, S, kT) ||
        !make_bf16_map(&tu, p.U, D, p.m, p.heads, kMP) || !make_bf16_map(&th, p.H, D, p.n, S, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(anchor_causal_wide_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
    if (e != cudaSuccess) return e;
    CwParams cp;
    cp.heads = p.heads;
    cp.n = p.n;
    cp.m = p.m;
    cp.tiles = (p.n + kT - 1) / kT;
    cp.chunks = causal_wide_chunks(S, cp.tiles);
    cp.c = p.scale * 1.4426950408889634f;
    cp.H = static_cast<__nv_bfloat16 *>(p.H);
    cp.wait_ns = 2000000000ull;
    return launch_pdl(anchor_causal_wide_kernel<D>, dim3((unsigned)(S * cp.chunks)), dim3(kThreads), LY::kSmem, stream,
                      tq, tv, tu, th, cp);
}

}  // namespace

// bf16, d = 128 with any m <= 128, or d = 64 with 64 < m <= 128 (the 64-anchor kernel takes
// d = 64, m <= 64)
bool causal_wide_supported(const Problem &p) {
    return !p.f32 && p.m >= 1 && p.m <= kMP && p.n >= 1 && (p.d == 128 || (p.d == 64 && p.m > 64));
}

cudaError_t launch_causal_wide(const Problem &p, cudaStream_t stream) {
    if (p.d == 128) return launch_d<128>(p, stream);
    if (p.d == 64) return launch_d<64>(p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t causal_wide_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_causal_wide_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_causal_wide_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

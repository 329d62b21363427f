// Backward of the anchor-attention forward on the tensor cores for d = 128 and m <= 128 (bf16
// operands, fp32 accumulators in tensor memory), any n.  For an upstream gradient dH of
// H = A Delta^{-1} (A^T V), A = rowsoftmax(scale Q U^T):
//   dW' = A^T dH,  dW = Delta^{-1} dW',  dDelta_j = -sum_k dW_jk W'_jk,
//   G = dH W'^T + V dW^T + 1 dDelta^T,  dS = A o (G - rowsum(A o G)),
//   dQ = scale dS U,  dV = A dW,  dU = scale dS^T Q summed over the batch entries of a head
// (the anchors are fitted by gradient descent: pith.science verdict on arXiv 2505.16463,
// "core_discovery"; the arXiv abstract, where the anchors are weights of a trainable layer).
//
// At d = m = 128 one CTA cannot hold a slice's whole backward (the four W', dW images alone
// take 128 KB of shared memory, and the accumulators S, G, dQ, dV and dU 640 tensor-memory
// columns), so the work runs as four launches over items (a slice's run of consecutive 128-token
// tiles; the chunking depends on the shape alone, so the sums and the bits do too):
//   pass 1   S_t = Q_t U^T, A_t = softmax; W += A_t^T V_t, then [dW' | Delta] +=
//            A_t^T [dH_t | 1] (one N = 144 product), with A as hi + lo bf16 parts released
//            one after the other; Q, V, dH in buffers of their own, each refilled by its own
//            producer warp as soon as its products are done; the item's W, dW', Delta go to a
//            workspace row block
//   reduce   per slice: the items' blocks summed in order; W' = W / Delta, dW = dW' / Delta
//            as hi + lo bf16 images [4][128][128], and dDelta (fp32)
//   pass 2   S_t again and e = 2^(c s - M) (A = e / z); G_t = dH_t (W'_hi + W'_lo)^T +
//            V_t (dW_hi + dW_lo)^T with the images streamed through a two-slot ring (from L2:
//            every item of a slice reads the same 128 KB); dS_t on CUDA cores in fp32;
//            dV_t = e dW (scaled by 1/z on the way out), dU += dS_t^T Q_t, dQ_t = dS_hi U;
//            the item's dU to a workspace block
//   dU sum   per head, the items' blocks in (batch entry, item) order (the backward's dU
//            kernel)
// The fp32 operands that the gradients sum over many terms - A in pass 1, W' and dW in G, dS
// in dU - enter the MMAs as two bf16 parts, hi = bf16(x) and lo = bf16(x - hi): with any one of
// them rounded once to bf16, dU of the 16384-token workload (four batch entries) comes out at
// 0.8 to 1.1 of the bf16 tolerance in a float64 emulation; with all of them split at 0.003
// (dQ, a sum over the m anchors only, stays at 0.06 with dS_hi alone).
// Pass 2's shared memory (U | Q | dQ, dV staging | V or dS_hi | dH or dS_lo | image ring) fills
// 224 KB: dS_t is written over V_t and dH_t once G_t is done, and e (bf16) over S_t in tensor
// memory, where dV_t reads it.  Tensor memory (512 columns): S then e | G then dQ | dV | dU.
// Warps: row warps 0-7 (warp w: TMEM lanes 32 (w % 4) .. + 31, tokens or anchors for the
// item's sums; half w / 4 of the columns, the halves' row sums exchanged through shared or
// tensor memory), then the producer warps and the MMA warp (see kP1Issue, kP2Issue).  Every
// wait is bounded; one that gives up sets bit 0 of the error word and the CTA drains what it
// has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"
#include "tmem_pair.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_bwd_wide_error;  // bit 0: a pipeline wait gave up

namespace {

using namespace ptx;

constexpr int kT = 128, kMP = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kBlkB = kT * 128;   // one 64-column block of a 128-row bf16 tile (16 KB)
constexpr int kAB = kT * kMP * 2; // a [128 tokens][128 anchors] bf16 tile (A, dS: 32 KB)
constexpr int kStageB = 8 * 4096; // pass 2's dQ / dV staging: 4 KB per row warp
constexpr int k1Bars = 15, k2Bars = 27;
// row warps 0-7 in both passes (two per TMEM lane quarter, one per half of the columns), then
// producer warps (one per input in pass 1: Q, V, dH; in pass 2 one for Q, dH, V and one for the
// image ring: a lane that sleeps in an mbarrier wait holds up its whole warp), then the MMA warp
constexpr int kRowWarps = 8, kWarpProd = kRowWarps;
constexpr int kP1Threads = 32 * (kRowWarps + 4), kP1Issue = kRowWarps + 3;
constexpr int kP2Threads = 32 * (kRowWarps + 3), kP2Issue = kRowWarps + 2;
constexpr uint32_t k1ColS = 0, k1ColWD = 128;
constexpr uint32_t k2ColS = 0, k2ColG = 128, k2ColDV = 256, k2ColDU = 384;  // dQ_t reuses G's columns

// Sizes and shared-memory layouts for head dimension D (64 or 128).
template <int D>
struct Geo {
    static constexpr int kNB = D / 64;               // 64-column blocks of a [rows][D] tile
    static constexpr int kQB = kT * D * 2;           // a [128 tokens][D] bf16 tile (Q, V, dH)
    static constexpr int kUB = kMP * D * 2;          // a [128 anchors][D] bf16 tile (U, an image)
    static constexpr int kPartF = kMP * 2 * D + kMP; // an item's pass-1 block: [W | dW'] rows, then Delta
    static constexpr uint32_t k1ColDelta = k1ColWD + 2 * D;
    // pass 1: U | Q | V | dH | ones [128][64] (dH's block after its last: [dH | 1] is one
    // N = D + 16 operand) | A_hi | A_lo | row-sum exchange [2][128] | barriers
    static constexpr int k1U = 0, k1Q = k1U + kUB, k1V = k1Q + kQB, k1H = k1V + kQB, k1Ones = k1H + kQB;
    static constexpr int k1AH = k1Ones + kBlkB, k1AL = k1AH + kAB, k1Ex = k1AL + kAB, k1Bar = k1Ex + 2 * kT * 8;
    static constexpr int k1Smem = k1Bar + k1Bars * 8 + 16 + 1024;
    // pass 2: U | Q | dQ, dV staging | V or dS_hi | dH or dS_lo | image ring (2 slots) | dDelta |
    // barriers (V and dH each sit at the start of a 32 KB dS tile)
    static constexpr int k2U = 0, k2X = k2U + kUB, k2Stage = k2X + kQB, k2VH = k2Stage + kStageB;
    static constexpr int k2Img = k2VH + 2 * kAB, k2DD = k2Img + 2 * kUB, k2Bar = k2DD + kMP * 4;
    static constexpr int k2Smem = k2Bar + k2Bars * 8 + 16 + 1024;
    static_assert(k1Smem <= 227 * 1024 && k2Smem <= 227 * 1024, "shared memory");
    static_assert(k1ColWD + 2 * D + 16 <= kTmemCols, "tensor memory");
};

struct BwParams {
    int heads, n, m, tiles, chunks;
    float c;      // scale * log2(e)
    float scale;
    float *part;           // pass 1: [slices * chunks][kPartF of D]
    const float *ddelta;   // pass 2: [slices][kMP]
    float *dupart;         // pass 2: [slices][chunks][m][D]
    __nv_bfloat16 *dQ, *dV;
    uint64_t wait_ns;
};

// byte offset of 16-byte chunk c (0..15) of row r in a swizzled [rows][128] bf16 tile stored as
// two 64-column blocks of rows x 128 bytes (the layout a TMA load of the tile produces)
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// descriptor advance for K step kk (16 elements) of a K-major [128 rows][128] swizzled tile
__device__ __forceinline__ uint64_t kstep(int kk) { return (uint64_t)((((kk >> 2) * kT * 128) + (kk & 3) * 32) >> 4); }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8(const float *x, float r) {
    return make_uint4(pack2(x[0] * r, x[1] * r), pack2(x[2] * r, x[3] * r), pack2(x[4] * r, x[5] * r),
                      pack2(x[6] * r, x[7] * r));
}
// bf16 parts of 8 floats: hi = round(x), lo = round(x - hi) (hi read back from its packed pair:
// the low bf16 of a pair is the even element)
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        h[k] = pack2(x[2 * k], x[2 * k + 1]);
        const float h0 = __uint_as_float(h[k] << 16), h1 = __uint_as_float(h[k] & 0xffff0000u);
        l[k] = pack2(x[2 * k] - h0, x[2 * k + 1] - h1);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t par, uint64_t limit_ns) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, par, 2000)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_bwd_wide_error, 1u);
            return false;
        }
    }
    return true;
}

// the TMA boxes (64 columns each) of a [128][64 NB] bf16 tile
template <int NB>
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int row, int outer,
                                          uint64_t pol) {
#pragma unroll
    for (int b = 0; b < NB; ++b) tma_load_3d(dst + b * kBlkB, map, bar, 64 * b, row, outer, pol);
}

// an L2 prefetch of the boxes of a [128][64 NB] bf16 tile (no shared memory, no completion):
// the kernels keep one tile of each input in shared memory, so the load of the next one is
// issued late and would otherwise wait out the full memory latency
template <int NB>
__device__ __forceinline__ void prefetch_tile(const CUtensorMap *map, int row, int outer) {
#pragma unroll
    for (int c0 = 0; c0 < 64 * NB; c0 += 64)
        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(c0), "r"(row), "r"(outer)
                     : "memory");
}

// the item's tiles: [t0, t1) of slice `slice` (chunks of balanced integer length)
struct Item {
    int slice, chunk, t0, nt;
};
__device__ __forceinline__ Item item_of(int b, int tiles, int chunks) {
    Item it;
    it.slice = b / chunks;
    it.chunk = b - it.slice * chunks;
    it.t0 = (int)((long long)it.chunk * tiles / chunks);
    it.nt = (int)((long long)(it.chunk + 1) * tiles / chunks) - it.t0;
    return it;
}

// ------------------------------------------------------------------------------ pass 1
template <int D>
__global__ void __launch_bounds__(kP1Threads, 1)
anchor_bwd_wide_p1_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tdh, const __grid_constant__ CUtensorMap tu,
                          const BwParams p) {
    using GE = Geo<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + GE::k1Bar);
    uint64_t *u_full = bars + 0, *q_full = bars + 1, *q_empty = bars + 2, *v_full = bars + 3, *v_empty = bars + 4;
    uint64_t *h_full = bars + 5, *h_empty = bars + 6, *s_full = bars + 7, *a_full = bars + 8, *a_empty = bars + 9;
    uint64_t *acc_full = bars + 10, *mma_done = bars + 11, *x_ex = bars + 12, *al_full = bars + 13,
             *al_empty = bars + 14;  // a_full / a_empty: A_hi's
    float2 *s_mz = reinterpret_cast<float2 *>(sm + GE::k1Ex);  // [2][128]: each column half's (max, sum)
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + k1Bars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Item it = item_of(blockIdx.x, p.tiles, p.chunks);
    const int h = it.slice % p.heads;

    if (threadIdx.x == 0) {
        mbar_init(u_full, 1);
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(h_full, 1);
        mbar_init(h_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(a_full, kRowWarps);
        mbar_init(al_full, kRowWarps);
        mbar_init(al_empty, 1);
        mbar_init(x_ex, kRowWarps);
        mbar_init(a_empty, 1);
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == kP1Issue) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t sbase = smem_u32(sm);
    // launched with programmatic stream serialization: global memory only from here on
    grid_dependency_wait();
    grid_dependents_launch();

    if (warp >= kWarpProd && warp < kP1Issue) {
        // one warp per input (U and Q, V, dH), so that no refill waits behind another
        if (lane == 0) {
            const int w = warp - kWarpProd;
            const uint64_t pol_keep = policy_evict_last();
            const CUtensorMap *map = w == 0 ? &tq : (w == 1 ? &tv : &tdh);
            uint64_t *full = w == 0 ? q_full : (w == 1 ? v_full : h_full);
            uint64_t *empty = w == 0 ? q_empty : (w == 1 ? v_empty : h_empty);
            uint8_t *dst = sm + (w == 0 ? GE::k1Q : (w == 1 ? GE::k1V : GE::k1H));
            tma_prefetch_desc(map);
            if (w == 0) {
                tma_prefetch_desc(&tu);
                mbar_arrive_expect_tx(u_full, GE::kUB);
                load_tile<GE::kNB>(sm + GE::k1U, &tu, u_full, 0, h, pol_keep);
            }
            int n = 0;
            for (int i = 0; i < it.nt; ++i) {
                const int row = (it.t0 + i) * kT;
                // this input's tiles two ahead (and, at the start, the next) into L2
                for (int k = i == 0 ? 1 : 2; k <= 2; ++k)
                    if (i + k < it.nt) prefetch_tile<GE::kNB>(map, row + k * kT, it.slice);
                if (i >= 1 && !bwait(empty, (uint32_t)((i - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(full, GE::kQB);
                load_tile<GE::kNB>(dst, map, full, row, it.slice, pol_keep);
                ++n;
            }
            // the CTA leaves only once its copies have landed
            if (n > 0) bwait(full, (uint32_t)((n - 1) & 1), p.wait_ns);
            if (w == 0) bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kP1Issue) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);       // [tokens x anchors], K = d
            const uint32_t idW = idesc_bf16_f32(kMP, D, true, true);          // A^T V, K = tokens
            const uint32_t idWD = idesc_bf16_f32(kMP, D + 16, true, true);    // A^T [dH | 1]
            const uint64_t udesc = smem_desc_sw128(sbase + GE::k1U, 16, 1024);
            const uint64_t qdesc = smem_desc_sw128(sbase + GE::k1Q, 16, 1024);
            const uint64_t vdesc = smem_desc_sw128(sbase + GE::k1V, kBlkB, 1024);
            const uint64_t hdesc = smem_desc_sw128(sbase + GE::k1H, kBlkB, 1024);  // dH | ones
            bool ok = bwait(u_full, 0u, p.wait_ns);
            auto issue_s = [&](int i) -> bool {
                if (!bwait(q_full, (uint32_t)(i & 1), p.wait_ns)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_bf16(tmem + k1ColS, qdesc + kstep(kk), udesc + kstep(kk), idS, kk > 0 ? 1u : 0u);
                umma_commit(s_full);
                umma_commit(q_empty);
                return true;
            };
            if (ok && it.nt > 0) ok = issue_s(0);
            for (int i = 0; i < it.nt && ok; ++i) {
                // the row warps have read S_i and written A_hi of tile i
                if (!bwait(a_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                if (i + 1 < it.nt && !issue_s(i + 1)) { ok = false; break; }
                // W += A_hi^T V + A_lo^T V (then V's buffer is refilled), [dW' | Delta] +=
                // A_hi^T [dH | 1] (then A_hi's buffer takes the next tile's) + A_lo^T [dH | 1]
                const uint64_t ahd = smem_desc_sw128(sbase + GE::k1AH, kBlkB, 1024);  // A^T, MN-major
                const uint64_t ald = smem_desc_sw128(sbase + GE::k1AL, kBlkB, 1024);
                if (!bwait(v_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + k1ColWD, ahd + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), idW,
                              (i > 0 || kt > 0) ? 1u : 0u);
                if (!bwait(al_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + k1ColWD, ald + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), idW, 1u);
                umma_commit(v_empty);
                if (!bwait(h_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + k1ColWD + D, ahd + (uint64_t)(kt * 128), hdesc + (uint64_t)(kt * 128), idWD,
                              (i > 0 || kt > 0) ? 1u : 0u);
                umma_commit(a_empty);
#pragma unroll
                for (int kt = 0; kt < kT / 16; ++kt)
                    umma_bf16(tmem + k1ColWD + D, ald + (uint64_t)(kt * 128), hdesc + (uint64_t)(kt * 128), idWD, 1u);
                umma_commit(al_empty);
                umma_commit(h_empty);
            }
            if (ok) umma_commit(acc_full);
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (tokens; anchors for the item's sums), column
        // group g = w / 4 (anchors 64 g .. 64 g + 63; W or dW' for the item's sums)
        const int row = (warp & 3) * 32 + lane, g = warp >> 2;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        {   // the ones block (every element 1; the MMA reads its first 16 columns)
            const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
            for (int i = warp * 32 + lane; i < kBlkB / 16; i += 32 * kRowWarps) reinterpret_cast<uint4 *>(sm + GE::k1Ones)[i] = ones;
        }
        bool ok = true;
        float e[64];
        for (int i = 0; i < it.nt && ok; ++i) {
            const bool valid = (it.t0 + i) * kT + row < p.n;
            if (!bwait(s_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            // this half's maximum, exponentials and sum; the halves' (max, sum) exchanged, and
            // both scaled to the row's maximum: A_j = e_j 2^(m_g - M) / (z_0 2^(m_0 - M) + z_1 2^(m_1 - M))
            float mg;
            {
                tmem_ld32(trow + k1ColS + 64 * g, e);
                tmem_ld32(trow + k1ColS + 64 * g + 32, e + 32);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 64; ++j) e[j] = 64 * g + j < p.m ? e[j] * p.c : -INFINITY;
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = e[k];
#pragma unroll
                for (int j = 8; j < 64; j += 8)
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], e[j + k]);
                mg = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                // a half with every anchor masked (m <= 64) has no maximum: its terms are zero
                const float ms = mg == -INFINITY ? 0.f : mg;
#pragma unroll
                for (int j = 0; j < 64; ++j) e[j] = rowops::ex2_approx(e[j] - ms);
            }
            float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 64; ++j) z4[j & 3] += e[j];
            s_mz[g * kT + row] = make_float2(mg, (z4[0] + z4[1]) + (z4[2] + z4[3]));
            __syncwarp();
            if (lane == 0) mbar_arrive(x_ex);
            if (!bwait(x_ex, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
            const float2 h0 = s_mz[row], h1 = s_mz[kT + row];
            const float M = fmaxf(h0.x, h1.x);  // finite: half 0 holds anchor 0
            const float f0 = h0.x == -INFINITY ? 0.f : rowops::ex2_approx(h0.x - M);
            const float f1 = h1.x == -INFINITY ? 0.f : rowops::ex2_approx(h1.x - M);
            const float z = h0.y * f0 + h1.y * f1;
            const float zinv = valid ? (g == 0 ? f0 : f1) / z : 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) e[j] *= zinv;
            uint4 hi[8], lo[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) split8(e + 8 * c, hi[c], lo[c]);
            // A_hi once the previous tile's products have read it, then A_lo likewise
            if (i >= 1 && !bwait(a_empty, (uint32_t)((i - 1) & 1), p.wait_ns)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(sm + GE::k1AH + sw_off(row, 8 * g + c, kT)) = hi[c];
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
            if (i >= 1 && !bwait(al_empty, (uint32_t)((i - 1) & 1), p.wait_ns)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(sm + GE::k1AL + sw_off(row, 8 * g + c, kT)) = lo[c];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(al_full);
        }
        // the item's W | dW' | Delta: anchor j = row; group 0 W and Delta, group 1 dW'
        ok = ok && it.nt > 0 && bwait(acc_full, 0u, p.wait_ns);
        if (ok) {
            tc_fence_after();
            float *dst = p.part + (size_t)blockIdx.x * GE::kPartF;
            float o[32];
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
                tmem_ld32(trow + k1ColWD + D * g + 32 * q, o);
                tmem_ld_wait();
                float4 *d4 = reinterpret_cast<float4 *>(dst + (size_t)row * 2 * D + D * g + 32 * q);
#pragma unroll
                for (int k = 0; k < 8; ++k) d4[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
            }
            if (g == 0) {
                tmem_ld32(trow + GE::k1ColDelta, o);
                tmem_ld_wait();
                dst[kMP * 2 * D + row] = o[0];
            }
            tc_fence_before();
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == kP1Issue) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------------ reduce
// Per slice and run of kRJ anchors (one CTA of D threads; thread k = column k): W, dW' and Delta summed over
// the slice's items in item order; W' = W / Delta and dW = dW' / Delta as hi + lo bf16 images
// (rows >= m and anchors with Delta = 0 are zero), dDelta_j = -sum_k dW_jk W'_jk in fp32 (a
// fixed warp tree, then the warps in order).
constexpr int kRJ = 8;
template <int D>
__global__ void __launch_bounds__(D)
anchor_bwd_wide_reduce_kernel(const float *__restrict__ part, int chunks, int m, __nv_bfloat16 *__restrict__ img,
                              float *__restrict__ ddelta) {
    constexpr int kPartF = Geo<D>::kPartF;
    __shared__ float s_red[D / 32][kRJ];
    __shared__ float s_rinv[kRJ];
    grid_dependency_wait();
    grid_dependents_launch();
    const int slice = blockIdx.x, j0 = blockIdx.y * kRJ, k = threadIdx.x, lane = k & 31, warp = k >> 5;
    const float *P = part + (size_t)slice * chunks * kPartF;
    float w[kRJ], dw[kRJ], dl[kRJ];
#pragma unroll
    for (int r = 0; r < kRJ; ++r) w[r] = dw[r] = dl[r] = 0.f;
    for (int c = 0; c < chunks; ++c) {
        const float *pc = P + (size_t)c * kPartF;
#pragma unroll
        for (int r = 0; r < kRJ; ++r) {
            w[r] = __fadd_rn(w[r], __ldg(pc + (size_t)(j0 + r) * 2 * D + k));
            dw[r] = __fadd_rn(dw[r], __ldg(pc + (size_t)(j0 + r) * 2 * D + D + k));
            dl[r] = __fadd_rn(dl[r], __ldg(pc + kMP * 2 * D + j0 + r));
        }
    }
    __nv_bfloat16 *I = img + (size_t)slice * 4 * kMP * D;
#pragma unroll
    for (int r = 0; r < kRJ; ++r) {
        const int j = j0 + r;
        const float rinv = (j < m && dl[r] != 0.f) ? 1.f / dl[r] : 0.f;
        if (k == 0) s_rinv[r] = rinv;
        const float wp = w[r] * rinv, dwv = dw[r] * rinv;
        const __nv_bfloat16 wh = __float2bfloat16_rn(wp), dh = __float2bfloat16_rn(dwv);
        I[(size_t)(0 * kMP + j) * D + k] = wh;
        I[(size_t)(1 * kMP + j) * D + k] = __float2bfloat16_rn(wp - __bfloat162float(wh));
        I[(size_t)(2 * kMP + j) * D + k] = dh;
        I[(size_t)(3 * kMP + j) * D + k] = __float2bfloat16_rn(dwv - __bfloat162float(dh));
        float pr = dwv * wp;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) pr += __shfl_xor_sync(0xffffffffu, pr, o);
        if (lane == 0) s_red[warp][r] = pr;
    }
    __syncthreads();
    if (k < kRJ) {
        float dd = s_red[0][k];
#pragma unroll
        for (int q = 1; q < D / 32; ++q) dd = __fadd_rn(dd, s_red[q][k]);
        const int j = j0 + k;
        ddelta[(size_t)slice * kMP + j] = s_rinv[k] != 0.f ? -dd : 0.f;
    }
}

// ------------------------------------------------------------------------------ pass 2
template <int D>
__global__ void __launch_bounds__(kP2Threads, 1)
anchor_bwd_wide_p2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tdh, const __grid_constant__ CUtensorMap tu,
                          const __grid_constant__ CUtensorMap timg, const __grid_constant__ CUtensorMap tdq,
                          const __grid_constant__ CUtensorMap tdv, const BwParams p) {
    using GE = Geo<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + GE::k2Bar);
    uint64_t *u_full = bars + 0, *q_full = bars + 1, *x_free = bars + 3,
             *s_free = bars + 5, *v_full = bars + 7, *v_free = bars + 8, *img_full = bars + 9 /* [2] */,
             *img_empty = bars + 11 /* [2] */, *s_full = bars + 13, *s_empty = bars + 14, *g_full = bars + 15,
             *g_empty = bars + 16, *a_full = bars + 17, *dv_full = bars + 18, *dv_empty = bars + 19,
             *ds_full = bars + 20, *dq_full = bars + 21, *du_full = bars + 22, *mma_done = bars + 23,
             *x_ex = bars + 24, *h_full = bars + 25, *h_free = bars + 26;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + k2Bars);
    float *sDD = reinterpret_cast<float *>(sm + GE::k2DD);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Item it = item_of(blockIdx.x, p.tiles, p.chunks);
    const int h = it.slice % p.heads;

    if (threadIdx.x == 0) {
        mbar_init(u_full, 1);
        for (int b = 0; b < 2; ++b) {

            mbar_init(img_full + b, 1);
            mbar_init(img_empty + b, 1);
        }
        mbar_init(q_full, 1);
        mbar_init(x_free, 1);
        mbar_init(s_free, 1);
        mbar_init(v_full, 1);
        mbar_init(v_free, 1);
        mbar_init(h_full, 1);
        mbar_init(h_free, 1);
        mbar_init(s_full, 1);
        mbar_init(s_empty, 8);
        mbar_init(g_full, 1);
        mbar_init(g_empty, 8);
        mbar_init(a_full, 8);
        mbar_init(dv_full, 1);
        mbar_init(dv_empty, 8);
        mbar_init(ds_full, 8);
        mbar_init(dq_full, 1);
        mbar_init(du_full, 1);
        mbar_init(mma_done, 1);
        mbar_init(x_ex, 8);
        fence_mbar_init();
    }
    if (warp == kP2Issue) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t sbase = smem_u32(sm);
    grid_dependency_wait();
    grid_dependents_launch();

    if (warp == kWarpProd) {
        if (lane == 0) {
            // Q_i once dU has read Q_{i-1}; dH_i once dU has read dS_lo of tile i - 1 over
            // dH_{i-1}; V_i once dQ and dU have read dS_hi over V_{i-1} (the tiles ahead are
            // prefetched to L2)
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdh);
            tma_prefetch_desc(&tu);
            tma_prefetch_desc(&tdq);
            tma_prefetch_desc(&tdv);
            const uint64_t pol_keep = policy_evict_last(), pol_once = policy_evict_first();
            mbar_arrive_expect_tx(u_full, GE::kUB);
            load_tile<GE::kNB>(sm + GE::k2U, &tu, u_full, 0, h, pol_keep);
            int nq = 0, nh = 0, nv = 0;
            for (int i = 0; i < it.nt; ++i) {
                const int row = (it.t0 + i) * kT;
                for (int k = i == 0 ? 1 : 2; k <= 2; ++k)
                    if (i + k < it.nt) {
                        prefetch_tile<GE::kNB>(&tq, row + k * kT, it.slice);
                        prefetch_tile<GE::kNB>(&tv, row + k * kT, it.slice);
                        prefetch_tile<GE::kNB>(&tdh, row + k * kT, it.slice);
                    }
                if (i >= 1 && !bwait(x_free, (uint32_t)((i - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(q_full, GE::kQB);
                load_tile<GE::kNB>(sm + GE::k2X, &tq, q_full, row, it.slice, pol_once);
                ++nq;
                if (i >= 1 && !bwait(h_free, (uint32_t)((i - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(h_full, GE::kQB);
                load_tile<GE::kNB>(sm + GE::k2VH + kAB, &tdh, h_full, row, it.slice, pol_once);
                ++nh;
                if (i >= 1 && !bwait(v_free, (uint32_t)((i - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(v_full, GE::kQB);
                load_tile<GE::kNB>(sm + GE::k2VH, &tv, v_full, row, it.slice, pol_once);
                ++nv;
            }
            if (nq > 0) bwait(q_full, (uint32_t)((nq - 1) & 1), p.wait_ns);
            if (nh > 0) bwait(h_full, (uint32_t)((nh - 1) & 1), p.wait_ns);
            if (nv > 0) bwait(v_full, (uint32_t)((nv - 1) & 1), p.wait_ns);
            bwait(u_full, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpProd + 1) {
        if (lane == 0) {
            // the images W'_hi, W'_lo, dW_hi, dW_lo of every tile (unit u = 4 i + part, slot u & 1)
            tma_prefetch_desc(&timg);
            const uint64_t pol_keep = policy_evict_last();
            int nimg[2] = {0, 0};
            for (int u = 0; u < 4 * it.nt; ++u) {
                const int s = u & 1;
                if (u >= 2 && !bwait(img_empty + s, (uint32_t)(((u >> 1) - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(img_full + s, GE::kUB);
                load_tile<GE::kNB>(sm + GE::k2Img + s * GE::kUB, &timg, img_full + s, 0, it.slice * 4 + (u & 3), pol_keep);
                ++nimg[s];
            }
            for (int b = 0; b < 2; ++b)
                if (nimg[b] > 0) bwait(img_full + b, (uint32_t)((nimg[b] - 1) & 1), p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kP2Issue) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kT, kMP, false, false);  // [tokens x anchors], K = d
            const uint32_t idR = idesc_bf16_f32(kT, D, false, true);    // [tokens x d], K = anchors
            const uint32_t idU = idesc_bf16_f32(kMP, D, true, true);    // dS^T Q: anchors x d, K = tokens
            const uint64_t udesc = smem_desc_sw128(sbase + GE::k2U, 16, 1024);      // U, K-major (N = anchors)
            const uint64_t umn = smem_desc_sw128(sbase + GE::k2U, kBlkB, 1024);     // U, MN-major (N = d)
            const uint64_t vk = smem_desc_sw128(sbase + GE::k2VH, 16, 1024);
            const uint64_t hk = smem_desc_sw128(sbase + GE::k2VH + kAB, 16, 1024);
            bool ok = bwait(u_full, 0u, p.wait_ns);
            for (int i = 0; i < it.nt && ok; ++i) {
                const uint32_t xq = sbase + GE::k2X;
                // S_i = Q_i U^T, once dV_{i-1} has read A_{i-1} over S's columns
                if (!bwait(q_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                if (i >= 1 && !bwait(s_free, (uint32_t)((i - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint64_t qd = smem_desc_sw128(xq, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_bf16(tmem + k2ColS, qd + kstep(kk), udesc + kstep(kk), idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full);
                // G_i = dH_i (W'_hi + W'_lo)^T + V_i (dW_hi + dW_lo)^T, once dQ_{i-1} left G's columns
                if (!bwait(h_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                if (i >= 1 && !bwait(g_empty, (uint32_t)((i - 1) & 1), p.wait_ns)) { ok = false; break; }
                for (int part = 0; part < 4 && ok; ++part) {
                    const int u = 4 * i + part, s = u & 1;
                    if (part == 2 && !bwait(v_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                    if (!bwait(img_full + s, (uint32_t)((u >> 1) & 1), p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = part < 2 ? hk : vk;
                    const uint64_t bd = smem_desc_sw128(sbase + GE::k2Img + s * GE::kUB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_bf16(tmem + k2ColG, ad + kstep(kk), bd + kstep(kk), idS, (part > 0 || kk > 0) ? 1u : 0u);
                    if (part < 2) umma_commit(img_empty + s);  // W' parts: the slot takes a dW part next
                }
                if (!ok) break;
                umma_commit(g_full);
                // dV_i = A_i (dW_hi + dW_lo), A_i (bf16) in tensor memory over S's columns (the dW
                // parts are in slots 0 and 1)
                if (!bwait(a_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                if (i >= 1 && !bwait(dv_empty, (uint32_t)((i - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const uint64_t dwm = smem_desc_sw128(sbase + GE::k2Img + s * GE::kUB, kBlkB, 1024);
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16_tmem_a(tmem + k2ColDV, tmem + k2ColS + kj * 8, dwm + (uint64_t)(kj * 128), idR,
                                         (s > 0 || kj > 0) ? 1u : 0u);
                }
                umma_commit(dv_full);
                umma_commit(img_empty + 0);
                umma_commit(img_empty + 1);
                umma_commit(s_free);  // A_i read: S_{i+1} may be written there
                // dU += dS_lo^T Q_i first (dS_lo is over dH_i, whose buffer then takes dH_{i+1}),
                // then dU += dS_hi^T Q_i (Q's buffer then takes Q_{i+1}), then dQ_i = dS_hi U
                // (into G's columns; dQ sums over the m anchors only, so one bf16 part is enough;
                // V's buffer, under dS_hi, then takes V_{i+1})
                if (!bwait(ds_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint64_t qm = smem_desc_sw128(xq, kBlkB, 1024);  // Q_i, MN-major (N = d)
                    const uint64_t dsml = smem_desc_sw128(sbase + GE::k2VH + kAB, kBlkB, 1024);  // dS_lo^T
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt)
                        umma_bf16(tmem + k2ColDU, dsml + (uint64_t)(kt * 128), qm + (uint64_t)(kt * 128), idU,
                                  (i > 0 || kt > 0) ? 1u : 0u);
                    umma_commit(h_free);
                    const uint64_t dsk = smem_desc_sw128(sbase + GE::k2VH, 16, 1024);
                    const uint64_t dsm = smem_desc_sw128(sbase + GE::k2VH, kBlkB, 1024);  // dS_hi^T: anchors x tokens
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt)
                        umma_bf16(tmem + k2ColDU, dsm + (uint64_t)(kt * 128), qm + (uint64_t)(kt * 128), idU, 1u);
                    umma_commit(x_free);  // Q_i read: Q_{i+1} may load there
#pragma unroll
                    for (int kj = 0; kj < kMP / 16; ++kj)
                        umma_bf16(tmem + k2ColG, dsk + kstep(kj), umn + (uint64_t)(kj * 128), idR, kj > 0 ? 1u : 0u);
                }
                umma_commit(dq_full);
                umma_commit(v_free);
            }
            if (ok && it.nt > 0) umma_commit(du_full);
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ row warps
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (tokens; anchors for dU), column group
        // g = w / 4 (anchors, or d columns, 64 g .. 64 g + 63)
        const int row = (warp & 3) * 32 + lane, g = warp >> 2;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        if (g == 0) sDD[row] = p.ddelta[(size_t)it.slice * kMP + row];
        asm volatile("bar.sync 1, 256;" ::: "memory");
        bool ok = true;
        float e[64];          // 2^(c s_j - max) of this group's anchors (A = e / z)
        const uint64_t pol_out = policy_evict_first();
        float zinv_prev = 0.f;
        // dQ_i, then dV_i (as (e dW) / z): tensor memory -> this warp's staging [32 rows][64]
        // (swizzled like a TMA box) -> one TMA store of the warp's 32 rows and 64 columns (rows
        // past the slice are not written); the staging is reused once the previous store has
        // read it
        // (at D = 64 column half 0 drains all 64 columns, half 1 only arrives)
        uint8_t *stage = sm + GE::k2Stage + warp * 4096;
        const bool drains = D == 128 || g == 0;
        auto drain = [&](int i, uint64_t *full, uint64_t *empty, uint32_t col, const CUtensorMap *map,
                         float r) -> bool {
            if (!bwait(full, (uint32_t)(i & 1), p.wait_ns)) return false;
            tc_fence_after();
            float o[64];  // (at D = 64 half 1 reads columns past the tile's and stores nothing)
            tmem_ld32(trow + col + 64 * g, o);
            tmem_ld32(trow + col + 64 * g + 32, o + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(empty);
                bulk_wait_group_read0();
            }
            __syncwarp();
            if (drains) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(stage + sw_off(lane, c, 32)) = pack8(o + 8 * c, r);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(map, stage, 64 * g, (it.t0 + i) * kT + (warp & 3) * 32, it.slice, pol_out);
                    bulk_commit_group();
                }
            }
            return true;
        };
        auto drain_dq = [&](int i) -> bool { return drain(i, dq_full, g_empty, k2ColG, &tdq, p.scale); };
        auto drain_dv = [&](int i, float zinv) -> bool { return drain(i, dv_full, dv_empty, k2ColDV, &tdv, zinv); };
        for (int i = 0; i < it.nt && ok; ++i) {
            const bool valid = (it.t0 + i) * kT + row < p.n;
            // dQ and dV of the tile before first (dQ holds G's columns, which G_i needs, and the
            // rows would otherwise wait here for S_i)
            if (i >= 1 && !(drain_dq(i - 1) && drain_dv(i - 1, zinv_prev))) { ok = false; break; }
            if (!bwait(s_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            // this half's maximum, exponentials and sum; the halves' (max, sum) exchanged through
            // the last two of each half's own (already read) S columns, and e scaled to the row's
            // maximum M (both halves of dV's A operand must share it): A = e / z with
            // z = z_0 2^(m_0 - M) + z_1 2^(m_1 - M)
            float zinv;
            {
                tmem_ld32(trow + k2ColS + 64 * g, e);
                tmem_ld32(trow + k2ColS + 64 * g + 32, e + 32);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 64; ++j) e[j] = 64 * g + j < p.m ? e[j] * p.c : -INFINITY;
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = e[k];
#pragma unroll
                for (int j = 8; j < 64; j += 8)
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], e[j + k]);
                const float mg = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float ms = mg == -INFINITY ? 0.f : mg;  // a half with every anchor masked
#pragma unroll
                for (int j = 0; j < 64; ++j) e[j] = rowops::ex2_approx(e[j] - ms);
                float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 64; ++j) z4[j & 3] += e[j];
                const float2 mine = make_float2(mg, (z4[0] + z4[1]) + (z4[2] + z4[3]));
                tmem_st2(trow + k2ColS + 64 * g + 62, mine.x, mine.y);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_empty);  // this warp has read S_i and written its pair
                if (!bwait(s_empty, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                // (the other half's pair only: half 1 writes its A over half 0's pair columns
                // once it has read them)
                const float2 other = tmem_ld2(trow + k2ColS + 64 * (1 - g) + 62);
                tmem_ld_wait();
                const float2 h0 = g == 0 ? mine : other, h1 = g == 0 ? other : mine;
                const float M = fmaxf(h0.x, h1.x);  // finite: half 0 holds anchor 0
                const float f0 = h0.x == -INFINITY ? 0.f : rowops::ex2_approx(h0.x - M);
                const float f1 = h1.x == -INFINITY ? 0.f : rowops::ex2_approx(h1.x - M);
                const float fg = g == 0 ? f0 : f1;
#pragma unroll
                for (int j = 0; j < 64; ++j) e[j] *= fg;
                zinv = valid ? 1.f / (h0.y * f0 + h1.y * f1) : 0.f;
            }
            // e (bf16 pairs) over S's columns 32 g .. 32 g + 31 (dV's A operand)
            {
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) pk[j] = pack2(e[2 * j], e[2 * j + 1]);
                tmem_st32(trow + k2ColS + 32 * g, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
            // dS_j = A_j (G_j + dDelta_j - sum_l A_l (G_l + dDelta_l)), A = e / z, over V_i and dH_i
            if (!bwait(g_full, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            float gv[64];
            tmem_ld32(trow + k2ColG + 64 * g, gv);
            tmem_ld32(trow + k2ColG + 64 * g + 32, gv + 32);
            tmem_ld_wait();
            float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                gv[j] += sDD[64 * g + j];
                r4[j & 3] = fmaf(e[j], gv[j], r4[j & 3]);
            }
            const float rg = (r4[0] + r4[1]) + (r4[2] + r4[3]);
            // the two halves' r through tensor memory: each writes it into the first of its own
            // (already read) G columns and reads the other half's (G's columns take dQ_i only
            // after every row warp has passed ds_full)
            tmem_st2(trow + k2ColG + 64 * g, rg, 0.f);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(x_ex);
            if (!bwait(x_ex, (uint32_t)(i & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            const float2 other = tmem_ld2(trow + k2ColG + 64 * (1 - g));
            tmem_ld_wait();
            const float rr = g == 0 ? rg + other.x : other.x + rg;
            const float rs = rr * zinv;
#pragma unroll
            for (int j = 0; j < 64; ++j) gv[j] = e[j] * zinv * (gv[j] - rs);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 hi, lo;
                split8(gv + 8 * c, hi, lo);
                *reinterpret_cast<uint4 *>(sm + GE::k2VH + sw_off(row, 8 * g + c, kT)) = hi;
                *reinterpret_cast<uint4 *>(sm + GE::k2VH + kAB + sw_off(row, 8 * g + c, kT)) = lo;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
            zinv_prev = zinv;
        }
        if (ok && it.nt >= 1) ok = drain_dq(it.nt - 1) && drain_dv(it.nt - 1, zinv_prev);
        if (lane == 0) bulk_wait_group0();  // the stores have read the staging and landed
        __syncwarp();
        // the item's dU (scale dS^T Q): anchor j = row, d columns 64 g ..
        ok = ok && it.nt > 0 && bwait(du_full, 0u, p.wait_ns);
        if (ok) {
            tc_fence_after();
            float o[64];
            constexpr int DH = D / 2;  // this half's columns of dU
#pragma unroll
            for (int q = 0; q < DH / 32; ++q) tmem_ld32(trow + k2ColDU + DH * g + 32 * q, o + 32 * q);
            tmem_ld_wait();
            if (row < p.m) {
                float4 *dst = reinterpret_cast<float4 *>(p.dupart + ((size_t)blockIdx.x * p.m + row) * D + DH * g);
#pragma unroll
                for (int k = 0; k < DH / 4; ++k)
                    dst[k] = make_float4(o[4 * k] * p.scale, o[4 * k + 1] * p.scale, o[4 * k + 2] * p.scale,
                                         o[4 * k + 3] * p.scale);
            }
            tc_fence_before();
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == kP2Issue) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// items per slice: the split of the slice's tiles into `chunks` runs that keeps the most
// loaded SM's work (whole waves of kPlanSMs one-CTA-per-SM items, each its tiles plus about
// one tile's worth of setup and partial traffic) smallest; from the shape alone
int wide_chunks(long long slices, int tiles) {
    int best = 1;
    long long best_cost = -1;
    for (int c = 1; c <= tiles && c <= 64; ++c) {
        const long long waves = (slices * c + kPlanSMs - 1) / kPlanSMs;
        const long long cost = waves * ((tiles + c - 1) / c + 1);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

struct WideWs {
    size_t part = 0, img = 0, dd = 0, du = 0, total = 0;
};
WideWs wide_ws(const BwdProblem &p, int chunks) {
    auto up = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    const size_t S = (size_t)p.slices(), D = (size_t)p.d;
    WideWs w;
    w.part = 0;
    w.img = up(w.part + 4 * S * chunks * (kMP * 2 * D + kMP));
    w.dd = up(w.img + 2 * S * 4 * kMP * D);
    w.du = up(w.dd + 4 * S * kMP);
    w.total = w.du + 4 * S * chunks * (size_t)p.m * D;
    return w;
}

template <int D>
cudaError_t launch_wide(const BwdProblem &p, void *workspace, cudaStream_t stream) {
    using GE = Geo<D>;
    const long long S = p.slices();
    const int tiles = (p.n + kT - 1) / kT;
    const int chunks = wide_chunks(S, tiles);
    const WideWs L = wide_ws(p, chunks);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    CUtensorMap tq, tv, tdh, tu, timg, tdq, tdv;
    if (!make_bf16_map(&tq, p.Q, D, p.n, S, kT) || !make_bf16_map(&tv, p.V, D, p.n, S, kT) ||
        !make_bf16_map(&tdh, p.dH, D, p.n, S, kT) || !make_bf16_map(&tu, p.U, D, p.m, p.heads, kMP) ||
        !make_bf16_map(&timg, ws + L.img, D, kMP, S * 4, kMP) || !make_bf16_map(&tdq, p.dQ, D, p.n, S, 32) ||
        !make_bf16_map(&tdv, p.dV, D, p.n, S, 32))
        return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(anchor_bwd_wide_p1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, GE::k1Smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(anchor_bwd_wide_p2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, GE::k2Smem);
    if (e != cudaSuccess) return e;
    BwParams bp;
    bp.heads = p.heads;
    bp.n = p.n;
    bp.m = p.m;
    bp.tiles = tiles;
    bp.chunks = chunks;
    bp.c = p.scale * 1.4426950408889634f;
    bp.scale = p.scale;
    bp.part = reinterpret_cast<float *>(ws + L.part);
    bp.ddelta = reinterpret_cast<const float *>(ws + L.dd);
    bp.dupart = reinterpret_cast<float *>(ws + L.du);
    bp.dQ = static_cast<__nv_bfloat16 *>(p.dQ);
    bp.dV = static_cast<__nv_bfloat16 *>(p.dV);
    bp.wait_ns = 2000000000ull;
    const dim3 grid((unsigned)(S * chunks));
    if ((e = launch_pdl(anchor_bwd_wide_p1_kernel<D>, grid, dim3(kP1Threads), GE::k1Smem, stream, tq, tv, tdh, tu,
                        bp)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(anchor_bwd_wide_reduce_kernel<D>, dim3((unsigned)S, kMP / kRJ), dim3(D), 0, stream,
                        (const float *)bp.part, chunks, p.m, reinterpret_cast<__nv_bfloat16 *>(ws + L.img),
                        reinterpret_cast<float *>(ws + L.dd))) != cudaSuccess)
        return e;
    if ((e = launch_pdl(anchor_bwd_wide_p2_kernel<D>, grid, dim3(kP2Threads), GE::k2Smem, stream, tq, tv, tdh, tu, timg,
                        tdq, tdv, bp)) != cudaSuccess)
        return e;
    return launch_bwd_du_sum(bp.dupart, p.dU, p.B, p.heads, chunks, p.m * D, false, stream);
}

}  // namespace

bool bwd_wide_supported(const BwdProblem &p) {
    return !p.f32 && (p.d == 64 || p.d == 128) && p.m >= 1 && p.m <= kMP && p.n >= 1;
}

// d = 128 always; d = 64 when the one-CTA-per-slice kernel cannot take it (m > 64).  (At
// d = 64 with m <= 64 these kernels still pad the anchors to 128 and came out slower than the
// one-CTA-per-slice kernel even on long slices: 0.225 against 0.202 ms on 96 slices of 33 tiles.)
bool bwd_wide_preferred(const BwdProblem &p) {
    if (!bwd_wide_supported(p)) return false;
    return p.d == 128 || p.m > 64;
}

size_t bwd_wide_workspace(const BwdProblem &p) {
    return wide_ws(p, wide_chunks(p.slices(), (p.n + kT - 1) / kT)).total;
}

cudaError_t launch_bwd_wide(const BwdProblem &p, void *workspace, cudaStream_t stream) {
    return p.d == 64 ? launch_wide<64>(p, workspace, stream) : launch_wide<128>(p, workspace, stream);
}

cudaError_t bwd_wide_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_wide_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_bwd_wide_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

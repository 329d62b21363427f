// Anchor-attention forward for d = 64, m <= 64 with long slices, the slices' tiles split over
// a fixed number of CTAs (bf16 operands, fp32 accumulators in tensor memory).
//   H = A Delta^{-1} (A^T V), A = rowsoftmax(scale Q U^T), evaluated as A (Delta^{-1} (A^T V))
// (pith.science verdict on arXiv 2505.16463, "key_machinery" and the referee summary of
// Eq. 11/12).
//
// The G = slices x T tiles of 128 tokens, in slice-major order, are cut into kPlanSMs = 152
// contiguous ranges, one per CTA (the cut depends on the shape alone, so results do not
// depend on the device).  All CTAs are resident at once (a cooperative launch), which is what
// lets a CTA wait for the others that share one of its slices.  A CTA's range is a run of
// "parts", each the tiles of one slice that fall in the range.
//   Pass 1, part by part: S_t = Q_t U_h^T, A_t = softmax (row warps), [W | Delta] += A_t^T [V_t | 1]
//   into the part's tensor-memory accumulator; each A_t goes to a workspace by TMA (it stays
//   in L2).  At the end of a part two epilogue warps write its (W, Delta) partial to global
//   memory, each its half of the anchors; for each half, the last of the slice's parts to
//   arrive sums the slice's partials in part order, forms that half of W' = Delta^{-1} W as
//   the bf16 operand image and publishes it.
//   Pass 2, part by part: wait for the slice's W', load it and the part's A tiles back, and
//   form H_t = A_t W', stored by TMA.
// Warps: 0-7 row warps in two groups taking alternate tiles; 8 producer of Q (then of W' and
// A in pass 2) and of U; 9 MMA issuer; 10 producer of V; 12, 13 epilogue (TMEM lanes 0-63:
// the anchors).  Every wait, on this CTA's pipeline or on another CTA's partial, is bounded;
// one that gives up sets a bit of this kernel's error word (bit 0: the pipeline, bit 1: a
// slice's W'), and the CTA drains what it has in flight and leaves.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

#include <math.h>

namespace anchor {

__device__ unsigned int g_split_error;

namespace {

using namespace ptx;

constexpr int kT = 128, kD = 64, kMP = 64;
constexpr int kThreads = 448;
constexpr int kWarpQ = 8, kWarpMma = 9, kWarpV = 10, kWarpEpi = 12;
constexpr int kSlots = 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileB = kT * 64 * 2;   // a [128][64] bf16 tile (16 KB)
constexpr int kImgB = kMP * kD * 2;   // [64][64] bf16 (8 KB)
constexpr int kRowF = kD + 4;                 // a partial's anchor row: 64 W values, Delta, padding
constexpr int kPartFloats = kMP * kRowF;      // a (W, Delta) partial
// shared memory (an MN-major M = 128 operand reads an unused second 64-row block 16 KB on:
// A tile 1's is the first Q slot)
constexpr int kOffA = 0;                                // A tiles of the two row-warp groups
constexpr int kOffQRing = kOffA + 2 * kTileB;           // Q ring; in pass 2 the A tiles
constexpr int kOffVRing = kOffQRing + kSlots * kTileB;  // V ring; in pass 2 the H staging
constexpr int kOffOnes = kOffVRing + kSlots * kTileB;   // [128][64] bf16 ones: [V | 1]
constexpr int kOffU = kOffOnes + kTileB;                // U images [2]
constexpr int kOffWI = kOffU + 2 * kImgB;               // W' images [2]
constexpr int kOffBar = kOffWI + 2 * kImgB;
constexpr int kBars = 4 * kSlots + 30;
constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
// tensor memory: S_g at 64 g, the parts' [W | Delta] accumulators at 128 + 80 b, H_g at 288 + 64 g
constexpr uint32_t kColS = 0, kColWP = 128, kColH = 288;

struct SpParams {
    int heads, n, m, T;
    long long G;          // tiles of all slices
    int parts;            // CTAs the tiles are cut over
    int maxparts;         // most parts any slice has
    float c;              // scale * log2(e)
    unsigned *done;       // [slices][2] partial halves arrived (anchors 0-31, 32-63)
    unsigned *ready;      // [slices] halves of W' published (2: ready)
    float *part;          // [slices][maxparts][64][68]
    uint8_t *wimg;        // [slices][8 KB] W' operand images
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
            atomicOr(&g_split_error, 1u);
            return false;
        }
    }
    return true;
}

// The cut: CTA c takes global tiles [first(c), first(c + 1)) (G >= parts, so none is empty);
// the CTA of global tile x.
__device__ __forceinline__ long long first_tile(const SpParams &p, int c) { return (long long)c * p.G / p.parts; }
__device__ __forceinline__ int cta_of(const SpParams &p, long long x) { return (int)(((x + 1) * p.parts - 1) / p.G); }

// Local tile i of this CTA: its slice, tile in the slice, part index within this CTA, and
// whether it opens / closes its part.
struct Tile {
    int slice, t, part;
    bool first, last;
};
__device__ __forceinline__ Tile tile_at(const SpParams &p, long long x0, long long x1, long long i) {
    const long long x = x0 + i;
    Tile r;
    r.slice = (int)(x / p.T);
    r.t = (int)(x - (long long)r.slice * p.T);
    const long long s0 = x0 / p.T;
    r.part = (int)(r.slice - s0);
    r.first = i == 0 || r.t == 0;
    r.last = x + 1 == x1 || r.t == p.T - 1;
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
anchor_split_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap ta_st,
                    const __grid_constant__ CUtensorMap ta_ld, const __grid_constant__ CUtensorMap th,
                    const SpParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *qfull = bars, *qempty = qfull + kSlots, *vfull = qempty + kSlots, *vempty = vfull + kSlots;
    uint64_t *b2 = vempty + kSlots;  // pairs below: index 0/1
    uint64_t *s_full = b2, *s_empty = b2 + 2, *a_full = b2 + 4, *a_empty = b2 + 6, *h_full = b2 + 8,
             *h_empty = b2 + 10, *u_full = b2 + 12, *u_empty = b2 + 14, *wp_full = b2 + 16, *wp_empty = b2 + 18,
             *wi_full = b2 + 20, *wi_empty = b2 + 22;
    uint64_t *mma_done = b2 + 24, *astore = b2 + 25;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long x0 = first_tile(p, blockIdx.x), x1 = first_tile(p, blockIdx.x + 1);
    const int L = (int)(x1 - x0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(qfull + i, 1);
            mbar_init(qempty + i, 1);
            mbar_init(vfull + i, 1);
            mbar_init(vempty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(s_empty + i, 4);
            mbar_init(a_full + i, 4);
            mbar_init(a_empty + i, 1);
            mbar_init(h_full + i, 1);
            mbar_init(h_empty + i, 4);
            mbar_init(u_full + i, 1);
            mbar_init(u_empty + i, 1);
            mbar_init(wp_full + i, 1);
            mbar_init(wp_empty + i, 2);
            mbar_init(wi_full + i, 1);
            mbar_init(wi_empty + i, 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(astore, 8);
        fence_mbar_init();
    }
    if (warp < 8) {  // the ones block
        const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = threadIdx.x; i < kTileB / 16; i += 256) reinterpret_cast<uint4 *>(sm + kOffOnes)[i] = ones;
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t sbase = smem_u32(sm);

    if (warp == kWarpQ) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tu);
            tma_prefetch_desc(&ta_ld);
            const uint64_t pol_once = policy_evict_first(), pol_keep = policy_evict_last();
            int seq = 0, uloads = 0, wloads = 0;
            bool ok = true;
            // pass 1: each part's U, then its Q tiles
            for (int i = 0; i < L && ok; ++i) {
                const Tile tl = tile_at(p, x0, x1, i);
                if (tl.first) {
                    const int b = tl.part & 1;
                    if (tl.part >= 2 && !bwait(u_empty + b, (uint32_t)(((tl.part >> 1) - 1) & 1), p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(u_full + b, kImgB);
                    tma_load_3d(sm + kOffU + b * kImgB, &tu, u_full + b, 0, 0, tl.slice % p.heads, pol_keep);
                    ++uloads;
                }
                const int s = seq % kSlots;
                if (seq >= kSlots && !bwait(qempty + s, (uint32_t)(((seq / kSlots) - 1) & 1), p.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(qfull + s, kTileB);
                tma_load_3d(sm + kOffQRing + s * kTileB, &tq, qfull + s, 0, tl.t * kT, tl.slice, pol_once);
                ++seq;
            }
            // pass 2: each part's W' once its slice has published it, then its A tiles (every
            // A store of this CTA has completed: the row warps arrive on astore after theirs)
            ok = ok && bwait(astore, 0u, p.wait_ns);
            for (int i = 0; i < L && ok; ++i) {
                const Tile tl = tile_at(p, x0, x1, i);
                if (tl.first) {
                    const int b = tl.part & 1;
                    if (tl.part >= 2 && !bwait(wi_empty + b, (uint32_t)(((tl.part >> 1) - 1) & 1), p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t *flag = p.ready + tl.slice;
                    if (ld_acquire_gpu(flag) < 2u) {
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire_gpu(flag) < 2u) {
                            if (globaltimer_ns() - t0 > p.wait_ns) {
                                atomicOr(&g_split_error, 2u);
                                ok = false;
                                break;
                            }
                            __nanosleep(128);
                        }
                        if (!ok) break;
                    }
                    fence_proxy_async_global();
                    mbar_arrive_expect_tx(wi_full + b, kImgB);
                    bulk_load(sm + kOffWI + b * kImgB, p.wimg + (size_t)tl.slice * kImgB, kImgB, wi_full + b);
                    ++wloads;
                }
                const int s = seq % kSlots;
                if (seq >= kSlots && !bwait(qempty + s, (uint32_t)(((seq / kSlots) - 1) & 1), p.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(qfull + s, kTileB);
                tma_load_3d(sm + kOffQRing + s * kTileB, &ta_ld, qfull + s, 0, tl.t * kT, tl.slice, pol_once);
                ++seq;
            }
            // every load issued has landed before the CTA leaves
            for (int s = 0; s < kSlots; ++s) {
                const int loads = seq > s ? (seq - s + kSlots - 1) / kSlots : 0;
                if (loads > 0) bwait(qfull + s, (uint32_t)((loads - 1) & 1), p.wait_ns);
            }
            for (int b = 0; b < 2; ++b) {
                const int nu = uloads > b ? (uloads - b + 1) / 2 : 0, nw = wloads > b ? (wloads - b + 1) / 2 : 0;
                if (nu > 0) bwait(u_full + b, (uint32_t)((nu - 1) & 1), p.wait_ns);
                if (nw > 0) bwait(wi_full + b, (uint32_t)((nw - 1) & 1), p.wait_ns);
            }
        }
        __syncwarp();
    } else if (warp == kWarpV) {
        if (lane == 0) {
            tma_prefetch_desc(&tv);
            const uint64_t pol_once = policy_evict_first();
            int issued = 0;
            for (int i = 0; i < L; ++i) {
                const Tile tl = tile_at(p, x0, x1, i);
                const int s = i % kSlots;
                if (i >= kSlots && !bwait(vempty + s, (uint32_t)(((i / kSlots) - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(vfull + s, kTileB);
                tma_load_3d(sm + kOffVRing + s * kTileB, &tv, vfull + s, 0, tl.t * kT, tl.slice, pol_once);
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
            const uint32_t idWD = idesc_bf16_f32(kT, kD + 16, true, true);    // [W | Delta] += A^T [V | 1]
            const uint32_t idH = idesc_bf16_f32(kT, kD, false, true);         // H = A W'
            bool ok = true;
            auto issue_s = [&](int i) -> bool {
                const Tile tl = tile_at(p, x0, x1, i);
                const int s = i % kSlots, g = i & 1, b = tl.part & 1;
                if (!bwait(qfull + s, (uint32_t)((i / kSlots) & 1), p.wait_ns)) return false;
                if (i >= 2 && !bwait(s_empty + g, (uint32_t)(((i >> 1) - 1) & 1), p.wait_ns)) return false;
                if (tl.first && !bwait(u_full + b, (uint32_t)((tl.part >> 1) & 1), p.wait_ns)) return false;
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(sbase + kOffQRing + s * kTileB, 16, 1024);
                const uint64_t udesc = smem_desc_sw128(sbase + kOffU + b * kImgB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16(tmem + kColS + g * 64, qdesc + (uint64_t)(kk * 2), udesc + (uint64_t)(kk * 2), idS,
                              kk > 0 ? 1u : 0u);
                umma_commit(s_full + g);
                umma_commit(qempty + s);
                if (tl.last) umma_commit(u_empty + b);  // the part's U has served its last S
                return true;
            };
            for (int i = 0; i < 2 && i < L && ok; ++i) ok = issue_s(i);
            for (int i = 0; i < L && ok; ++i) {
                const Tile tl = tile_at(p, x0, x1, i);
                const int s = i % kSlots, g = i & 1, b = tl.part & 1;
                if (i + 2 < L && !issue_s(i + 2)) { ok = false; break; }
                if (!bwait(a_full + g, (uint32_t)((i >> 1) & 1), p.wait_ns) ||
                    !bwait(vfull + s, (uint32_t)((i / kSlots) & 1), p.wait_ns)) {
                    ok = false;
                    break;
                }
                if (tl.first && tl.part >= 2 &&
                    !bwait(wp_empty + b, (uint32_t)(((tl.part >> 1) - 1) & 1), p.wait_ns)) {
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
                    umma_bf16(tmem + kColWP + b * 80, adesc + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), idWD,
                              (!tl.first || kt > 0) ? 1u : 0u);
                umma_commit(a_empty + g);
                umma_commit(vempty + s);
                if (tl.last) umma_commit(wp_full + b);
            }
            // pass 2: H_t = A_t W' (the part's image), A in the Q ring after the pass-1 tiles
            for (int i = 0; i < L && ok; ++i) {
                const Tile tl = tile_at(p, x0, x1, i);
                const int seq = L + i, s = seq % kSlots, g = i & 1, b = tl.part & 1;
                if (!bwait(qfull + s, (uint32_t)((seq / kSlots) & 1), p.wait_ns)) { ok = false; break; }
                if (tl.first && !bwait(wi_full + b, (uint32_t)((tl.part >> 1) & 1), p.wait_ns)) { ok = false; break; }
                if (i >= 2 && !bwait(h_empty + g, (uint32_t)(((i >> 1) - 1) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint64_t adesc = smem_desc_sw128(sbase + kOffQRing + s * kTileB, 16, 1024);
                const uint64_t wdesc = smem_desc_sw128(sbase + kOffWI + b * kImgB, kMP * 128, 1024);
#pragma unroll
                for (int kj = 0; kj < kMP / 16; ++kj)
                    umma_bf16(tmem + kColH + g * 64, adesc + (uint64_t)(kj * 2), wdesc + (uint64_t)(kj * 128), idH,
                              kj > 0 ? 1u : 0u);
                umma_commit(h_full + g);
                umma_commit(qempty + s);
                if (tl.last) umma_commit(wi_empty + b);
            }
            umma_commit(mma_done);
            bwait(mma_done, 0u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == kWarpEpi || warp == kWarpEpi + 1) {
        // ------------------------------------------------------------------ epilogue: anchor j
        // Each warp owns half of the anchors (32 rows) of every partial: it writes its half,
        // counts it in the slice's counter for that half, and, if it was the slice's last half
        // of its kind, sums the slice's halves in part order and writes that half of the W'
        // image - after writing its next partial, so that a reduction never holds up a partial
        // that other CTAs may be waiting for.
        const int half = warp - kWarpEpi;
        const int j = half * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // sum the slice's halves (row j) in part order; write that half of the W' image
        auto reduce = [&](int sl, int np) {
            __threadfence();
            const float4 *src = reinterpret_cast<const float4 *>(p.part + ((size_t)sl * p.maxparts * kMP + j) * kRowF);
            float4 acc[17];
#pragma unroll
            for (int k = 0; k < 17; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < np; ++q) {
                const float4 *row = src + (size_t)q * kMP * (kRowF / 4);
#pragma unroll
                for (int k = 0; k < 17; ++k) {
                    const float4 x = __ldcg(row + k);
                    acc[k] = make_float4(__fadd_rn(acc[k].x, x.x), __fadd_rn(acc[k].y, x.y), __fadd_rn(acc[k].z, x.z),
                                         __fadd_rn(acc[k].w, x.w));
                }
            }
            float wrow[64];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                wrow[4 * k] = acc[k].x;
                wrow[4 * k + 1] = acc[k].y;
                wrow[4 * k + 2] = acc[k].z;
                wrow[4 * k + 3] = acc[k].w;
            }
            rowops::scale64(wrow, acc[16].x != 0.f ? 1.f / acc[16].x : 0.f);
            uint8_t *img = p.wimg + (size_t)sl * kImgB;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) *reinterpret_cast<uint4 *>(img + sw_off(j, c8, kMP)) = pack8(wrow + 8 * c8);
            fence_proxy_async_global();
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(p.ready + sl, 1u);  // both halves published: 2
        };
        bool ok = true;
        int part = -1, pend_slice = -1, pend_np = 0;
        for (int i = 0; i < L && ok; ++i) {
            const Tile tl = tile_at(p, x0, x1, i);
            if (!tl.last) continue;
            ++part;
            const int b = part & 1;
            const int cfirst = cta_of(p, (long long)tl.slice * p.T);
            const int np = cta_of(p, (long long)tl.slice * p.T + p.T - 1) - cfirst + 1;
            const int pi = (int)blockIdx.x - cfirst;
            if (!bwait(wp_full + b, (uint32_t)((part >> 1) & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            float w[64], dl[32];
            tmem_ld32(trow + kColWP + b * 80, w);
            tmem_ld32(trow + kColWP + b * 80 + 32, w + 32);
            tmem_ld32(trow + kColWP + b * 80 + 64, dl);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(wp_empty + b);
            float4 *dst = reinterpret_cast<float4 *>(p.part + (((size_t)tl.slice * p.maxparts + pi) * kMP + j) * kRowF);
#pragma unroll
            for (int k = 0; k < 16; ++k) dst[k] = make_float4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            dst[16] = make_float4(dl[0], 0.f, 0.f, 0.f);
            __syncwarp();
            unsigned last = 0;
            if (lane == 0) {
                __threadfence();
                last = atomicAdd(p.done + 2 * tl.slice + half, 1u) == (unsigned)(np - 1);
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            // the reduction this warp owes for the part before runs now, after this partial
            if (pend_slice >= 0) reduce(pend_slice, pend_np);
            pend_slice = last ? tl.slice : -1;
            pend_np = np;
        }
        if (ok && pend_slice >= 0) reduce(pend_slice, pend_np);
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------------ row warps
        const int g = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        uint8_t *sA = sm + kOffA + g * kTileB;
        const uint64_t pol_a = policy_evict_last(), pol_out = policy_evict_first();
        bool ok = true;
        float v[64];
        for (int i = g, k = 0; i < L && ok; i += 2, ++k) {
            const Tile tl = tile_at(p, x0, x1, i);
            if (!bwait(s_full + g, (uint32_t)(k & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColS + g * 64, v);
            tmem_ld32(trow + kColS + g * 64 + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty + g);
            const float z = rowops::softmax64_unnormalised(v, p.m, p.c);
            rowops::scale64(v, tl.t * kT + row < p.n ? 1.f / z : 0.f);
            if (k >= 1 && !bwait(a_empty + g, (uint32_t)((k - 1) & 1), p.wait_ns)) { ok = false; break; }
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) *reinterpret_cast<uint4 *>(sA + sw_off(row, c8, kT)) = pack8(v + 8 * c8);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(a_full + g);
                if (tl.t * kT + q * 32 < p.n) {
                    tma_store_3d(&ta_st, sA + q * 32 * 128, 0, tl.t * kT + q * 32, tl.slice, pol_a);
                    bulk_commit_group();
                }
            }
        }
        // every A store of this warp is complete and visible to the pass-2 loads
        if (lane == 0) {
            bulk_wait_group0();
            fence_proxy_async_global();
            mbar_arrive(astore);
        }
        __syncwarp();
        // pass 2: H tiles out, staged over the V ring
        uint8_t *stage = sm + kOffVRing + warp * 4096;
        for (int i = g, k = 0; i < L && ok; i += 2, ++k) {
            const Tile tl = tile_at(p, x0, x1, i);
            if (!bwait(h_full + g, (uint32_t)(k & 1), p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(trow + kColH + g * 64, v);
            tmem_ld32(trow + kColH + g * 64 + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(h_empty + g);
                bulk_wait_group_read0();  // the last store has read the staging
            }
            __syncwarp();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) *reinterpret_cast<uint4 *>(stage + sw_off(lane, c8, 32)) = pack8(v + 8 * c8);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && tl.t * kT + q * 32 < p.n) {
                tma_store_3d(&th, stage, 0, tl.t * kT + q * 32, tl.slice, pol_out);
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

// the same cut on the host: the most parts any slice is split into
int max_parts(long long slices, int T, int parts) {
    const long long G = slices * T;
    auto cta = [&](long long x) { return (int)(((x + 1) * parts - 1) / G); };
    int mx = 1;
    for (long long s = 0; s < slices; ++s) mx = std::max(mx, cta(s * T + T - 1) - cta(s * T) + 1);
    return mx;
}

struct SplitLayout {
    size_t header = 0, part = 0, wimg = 0, abuf = 0, total = 0;
    int maxparts = 0;
};

SplitLayout split_layout(const Problem &p) {
    SplitLayout L;
    const long long S = p.slices();
    const int T = (p.n + kT - 1) / kT;
    L.maxparts = max_parts(S, T, kPlanSMs);
    auto up = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    // the A tiles first: a device that cannot hold every CTA at once runs the one-CTA-per-slice
    // kernel on the same workspace, whose only buffer they are
    L.abuf = 0;
    L.header = up((size_t)S * p.n * kD * 2);
    L.part = L.header + up(12 * (size_t)S);
    L.wimg = up(L.part + 4 * (size_t)S * L.maxparts * kPartFloats);
    L.total = L.wimg + (size_t)S * kImgB;
    return L;
}

}  // namespace

bool split_supported(const Problem &p) { return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1; }

size_t split_workspace(const Problem &p) { return split_layout(p).total; }

// cudaErrorCooperativeLaunchTooLarge when this device cannot hold all kPlanSMs CTAs at once
cudaError_t launch_split(const Problem &p, void *workspace, cudaStream_t stream) {
    const SplitLayout L = split_layout(p);
    const long long S = p.slices();
    // fewer tiles than CTAs: some CTAs would have none, and a slice's parts would no longer be
    // the CTAs between its first and last tile's; one CTA per slice then
    if (S * ((p.n + kT - 1) / kT) < kPlanSMs) return launch_stream(p, workspace, stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    CUtensorMap tq, tv, tu, ta_st, ta_ld, th;
    if (!make_bf16_map(&tq, p.Q, kD, p.n, S, kT) || !make_bf16_map(&tv, p.V, kD, p.n, S, kT) ||
        !make_bf16_map(&tu, p.U, kD, p.m, p.heads, kMP) || !make_bf16_map(&ta_st, ws + L.abuf, kMP, p.n, S, 32) ||
        !make_bf16_map(&ta_ld, ws + L.abuf, kMP, p.n, S, kT) || !make_bf16_map(&th, p.H, kD, p.n, S, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(anchor_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, anchor_split_kernel, kThreads, kSmem)) !=
        cudaSuccess)
        return e;
    if ((long long)sms * per_sm < kPlanSMs) return cudaErrorCooperativeLaunchTooLarge;
    if ((e = cudaMemsetAsync(ws + L.header, 0, L.part - L.header, stream)) != cudaSuccess) return e;
    SpParams sp;
    sp.heads = p.heads;
    sp.n = p.n;
    sp.m = p.m;
    sp.T = (p.n + kT - 1) / kT;
    sp.G = S * sp.T;
    sp.parts = kPlanSMs;
    sp.maxparts = L.maxparts;
    sp.c = p.scale * 1.4426950408889634f;
    sp.done = reinterpret_cast<unsigned *>(ws + L.header);
    sp.ready = sp.done + 2 * S;
    sp.part = reinterpret_cast<float *>(ws + L.part);
    sp.wimg = ws + L.wimg;
    sp.wait_ns = 2000000000ull;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPlanSMs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, anchor_split_kernel, tq, tv, tu, ta_st, ta_ld, th, sp);
}

cudaError_t split_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_split_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_split_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

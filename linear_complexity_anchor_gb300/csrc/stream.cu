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
// With few slices of many tiles, a cluster of c CTAs takes each slice: its T tiles are cut
// into c contiguous ranges, one per CTA; each CTA sums its range's tiles in its own
// accumulator, and after pass 1 every CTA of the cluster adds the c partial sums [W | Delta]
// over distributed shared memory in rank order (each gets the same bits) before its pass 2.
// More SMs then stream: 8 slices of 16384 tokens run as 8 clusters of 8 CTAs (53 us, against
// 126 us on 8 SMs).
// Every wait is bounded; one that gives up sets bit 0 of this kernel's error word and the
// CTA drains what it has in flight and leaves.
#include "cluster.cuh"
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
// clusters: this CTA's partial sums [anchor][64 W + Delta, 68 floats] after the pass-2
// staging in the V ring (free once pass 1's W MMAs are done)
constexpr int kPartRow = 68 * 4, kPartB = kMP * kPartRow;
constexpr int kOffPart = kOffVRing + kRowWarps * 4096;
static_assert(kOffPart + kPartB <= kOffOnes, "partial sums inside the V ring");
constexpr int kBars = 4 * kSlots + 4 * kNG + 2 * kNG * 2 + 8;
constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kOffStage + kRowWarps * 4096 <= kOffOnes, "pass-2 staging inside the V ring");
// tensor memory: pass 1 S_g at 64 g and [W | Delta] after them; pass 2 (W read out by then)
// H of group g, buffer b at 64 (2 g + b)
constexpr uint32_t kColS = 0, kColW = 64 * kNG, kColDelta = kColW + 64, kColH = 0;
static_assert(kColDelta + 16 <= 512 && 64 * 2 * kNG <= 512, "tensor memory columns");

struct StParams {
    int heads, n, m, tiles;
    int cl_c;  // CTAs per slice (a cluster; 1: one CTA per slice, no cluster)
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

// Clusters (warps 0 and 1, anchor j = row): this CTA's partial sums [W | Delta] go to its
// shared memory; once every CTA of the cluster has written its own, the c partials are added
// in rank order (every CTA adds the same values in the same order) and W' = W / Delta is
// written as the pass-2 operand image.  False if the wait for the cluster gave up.
__device__ __forceinline__ bool cluster_w_prime(uint8_t *sm, uint64_t *x_ready, uint64_t *x_done, uint32_t trow,
                                                int row, int ncl, uint64_t wait_ns) {
    tc_fence_after();
    {
        float w[64], dl[32];
        tmem_ld32(trow + kColW, w);
        tmem_ld32(trow + kColW + 32, w + 32);
        tmem_ld32(trow + kColDelta, dl);
        tmem_ld_wait();
        float4 *dst = reinterpret_cast<float4 *>(sm + kOffPart + row * kPartRow);
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        dst[16] = make_float4(dl[0], 0.f, 0.f, 0.f);
    }
    tc_fence_before();
    const uint32_t ready = smem_u32(x_ready), done = smem_u32(x_done);
    for (int r = 0; r < ncl; ++r) cl::arrive_release(cl::map_shared(ready, (uint32_t)r));
    const uint64_t t0 = globaltimer_ns();
    while (!cl::test_wait_acquire(ready, 0u)) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > wait_ns) {
            atomicOr(&g_stream_error, 1u);
            return false;
        }
    }
    const uint32_t mine = smem_u32(sm + kOffPart) + (uint32_t)(row * kPartRow);
    // (a remote load takes a round trip across the GPC: each batch of loads is issued before
    // any of its values is used, so that the round trips overlap)
    float dx[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) dx[r] = r < ncl ? cl::ld_f32(cl::map_shared(mine + 256, (uint32_t)r)) : 0.f;
    float dsum = dx[0];
#pragma unroll
    for (int r = 1; r < 8; ++r)
        if (r < ncl) dsum += dx[r];
    const float rinv = dsum != 0.f ? 1.f / dsum : 0.f;
    // 32 columns at a time
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        float acc[32];
#pragma unroll 1
        for (int r = 0; r < ncl; ++r) {
            const uint32_t src = cl::map_shared(mine + 128 * half, (uint32_t)r);
            float4 x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = cl::ld_f4(src + 16 * i);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (r == 0) {
                    acc[4 * i] = x[i].x, acc[4 * i + 1] = x[i].y, acc[4 * i + 2] = x[i].z, acc[4 * i + 3] = x[i].w;
                } else {
                    acc[4 * i] += x[i].x, acc[4 * i + 1] += x[i].y, acc[4 * i + 2] += x[i].z, acc[4 * i + 3] += x[i].w;
                }
            }
        }
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
            *reinterpret_cast<uint4 *>(sm + kOffW + sw_off(row, 4 * half + c8, kMP)) = pack8(acc + 8 * c8, rinv);
    }
    fence_proxy_async_smem();
    // this CTA is done with the cluster's partial sums
    for (int r = 0; r < ncl; ++r) cl::arrive_release(cl::map_shared(done, (uint32_t)r));
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
    uint64_t *x_ready = u_full + 5, *x_done = u_full + 6;  // cluster: partials written / read
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.tiles;
    // this CTA's tiles of its slice: [v0, v0 + L) (all T with one CTA per slice)
    const int ncl = p.cl_c, rank = blockIdx.x % ncl, slice = blockIdx.x / ncl;
    const int h = slice % p.heads;
    const int v0 = (int)((long long)rank * T / ncl), L = (int)((long long)(rank + 1) * T / ncl) - v0;

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
        mbar_init(x_ready, 64 * ncl);
        mbar_init(x_done, 64 * ncl);
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
    if (ncl > 1) cl::sync_all();  // the peers' barriers are initialised
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
            for (int seq = 0; seq < 2 * L; ++seq) {
                const int s = seq % kSlots;
                if (seq >= kSlots && !bwait(empty + s, (uint32_t)(((seq / kSlots) - 1) & 1), p.wait_ns)) break;
                uint8_t *st = sm + kOffQRing + s * kTileB;
                if (seq < L) {
                    mbar_arrive_expect_tx(full + s, kTileB);
                    tma_load_3d(st, &tq, full + s, 0, (v0 + seq) * kT, slice, pol_once);
                } else {
                    // pass 2: every A tile has been stored (the row warps finish their stores
                    // before they arrive on wp_full)
                    if (seq == L && !bwait(wp_full, 0u, p.wait_ns)) break;
                    mbar_arrive_expect_tx(full + s, kTileB);
                    tma_load_3d(st, &ta_ld, full + s, 0, (v0 + seq - L) * kT, slice, pol_once);
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
            for (int t = 0; t < L; ++t) {
                const int s = t % kSlots;
                if (t >= kSlots && !bwait(vempty + s, (uint32_t)(((t / kSlots) - 1) & 1), p.wait_ns)) break;
                mbar_arrive_expect_tx(vfull + s, kTileB);
                tma_load_3d(sm + kOffVRing + s * kTileB, &tv, vfull + s, 0, (v0 + t) * kT, slice, pol_once);
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
            for (int t = 0; t < L && ok; ++t) {
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
            for (int t = 0; t < L && ok; ++t) {
                // H buffer (g, b) of tile t = g + kNG k: b = k & 1, its use number k >> 1
                const int seq = L + t, s = seq % kSlots, k = t / kNG, hb = 2 * (t % kNG) + (k & 1), u = k >> 1;
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
            for (int t = 0; t < L && ok; ++t) {
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
        for (int t = g, k = 0; t < L && ok; t += kNG, ++k) {
            const int tt = v0 + t;
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
            rowops::scale64(v, tt * kT + row < p.n ? 1.f / z : 0.f);
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
                if (tt * kT + q * 32 < p.n) {
                    tma_store_3d(&ta_st, sA + q * 32 * 128, 0, tt * kT + q * 32, slice, pol_a);
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
        if (ok && ncl > 1) {
            if (warp < 2) ok = cluster_w_prime(sm, x_ready, x_done, trow, row, ncl, p.wait_ns);
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(wp_full);
        } else if (ok) {
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
        for (int t = g, k = 0; t < L && ok; t += kNG, ++k) {
            const int hb = 2 * g + (k & 1), tt = v0 + t;
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
            if (lane == 0 && tt * kT + q * 32 < p.n) {
                tma_store_3d(&th, stage, 0, tt * kT + q * 32, slice, pol_out);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
        // the cluster's CTAs have read this CTA's partial sums (this CTA's shared memory must
        // outlive their reads)
        if (ncl > 1 && warp < 2) {
            const uint32_t a = smem_u32(x_done);
            const uint64_t t0 = globaltimer_ns();
            while (!cl::test_wait_acquire(a, 0u)) {
                __nanosleep(256);
                if (globaltimer_ns() - t0 > p.wait_ns) {
                    atomicOr(&g_stream_error, 1u);
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool stream_supported(const Problem &p) { return !p.f32 && p.d == kD && p.m >= 1 && p.m <= kMP && p.n >= 1; }

// CTAs per slice: c = 1 (no cluster) or a cluster of 2 to 8, chosen from the shape alone (so
// the result bits depend on the shape only) for a GB300's capacity: how many clusters of c of
// these CTAs it holds at once (a cluster's CTAs share a GPC, so c = 3 fits 46, not 152 / 3:
// cudaOccupancyMaxActiveClusters on a GB300), kPlanSMs for c = 1.  The fewest tiles per CTA
// wins, with a second wave counted in full and a cluster kernel costing kClusterTiles tiles
// more; clusters only up to kClusterSlices slices, and with four tiles or more per CTA.  Both
// limits are measured on a GB300: a cluster kernel takes about 20 to 35 us more than its tiles
// at the one-CTA rate, and once the one-CTA plan streams from many SMs more SMs do not help
// (8 slices of 16384 tokens: 53 us in clusters of 8, against 126 us; 32 slices of 8000 tokens:
// 38 us in clusters of 4, against 66 us; 80 slices of 16384 tokens: 143 us in clusters of 3
// over two slices, against about 126 us; 96 slices of 4200 tokens: 48 us in clusters of 5 over
// four slices, against 40 us).  A device that holds fewer clusters runs the same plan, in more
// waves.
constexpr int kClusterCap[9] = {0, kPlanSMs, 76, 46, 36, 28, 23, 15, 15};
constexpr double kClusterTiles = 24.0;
constexpr long long kClusterSlices = kPlanSMs / 4;

int stream_cluster(const Problem &p) {
    if (p.plan_cl_c > 0) return p.plan_cl_c;
    const long long S = p.slices(), T = (p.n + kT - 1) / kT;
    int best = 1;
    double best_cost = (double)((S + kPlanSMs - 1) / kPlanSMs) * (double)T;
    if (S > kClusterSlices) return best;
    for (int c = 2; c <= 8; ++c) {
        if (T < 4LL * c) break;
        const double cost = (double)((S + kClusterCap[c] - 1) / kClusterCap[c]) * ((double)T / c + kClusterTiles);
        if (cost < 0.97 * best_cost) {
            best = c;
            best_cost = cost;
        }
    }
    return best;
}

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
    const int cl = stream_cluster(p);
    if (cl < 1 || cl > 8) return cudaErrorInvalidValue;
    StParams sp;
    sp.heads = p.heads;
    sp.n = p.n;
    sp.m = p.m;
    sp.tiles = (p.n + kT - 1) / kT;
    sp.cl_c = cl;
    sp.c = p.scale * 1.4426950408889634f;
    sp.wait_ns = 2000000000ull;
    // programmatic stream serialization, and the cluster shape
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * cl));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)cl;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = cl > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, anchor_stream_kernel, tq, tv, tu, ta_st, ta_ld, th, sp);
}

cudaError_t stream_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_stream_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

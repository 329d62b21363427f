// Tensor-core (tcgen05 / UMMA) variant of the anchor-attention forward
//   A = rowsoftmax(scale * Q U^T),  Delta = diag(colsum A),  H = A (Delta^{-1} (A^T V))
// (AnchorFormer, arXiv 2505.16463; pith.science verdict: "key_machinery", "core_discovery"
// and the referee summary of Eq. 11/12: B^T V -> Delta^{-1}(B^T V) -> B(Delta^{-1} B^T V)).
//
// One persistent kernel per call.  Work is cut into items handed out in a fixed ticket
// order by an atomic counter:
//   P1(s, c)  pass 1 over token chunk c of slice s: per 128-token tile, S = Q U^T on the
//             tensor core (TMEM accumulator), row softmax in registers (one thread per
//             token), A tile -> shared memory as bf16, then W += A^T V and Delta += A^T 1
//             on the tensor core (both from the same rounded A).  The chunk's (W, Delta)
//             goes to a workspace partial.  The last chunk of a slice to finish sums the
//             partials in chunk order (fixed: the result does not depend on which CTA ran
//             what), forms W' = Delta^{-1} W as a bf16 operand image and publishes it.
//   P2(s, c)  pass 2 over token chunk c: waits for the slice's W', recomputes A exactly as
//             P1 did, H = A W' on the tensor core, TMA store of the bf16 tile.
//   FULL(s)   short slices: P1 and P2 of a whole slice in one CTA, W' kept on chip.
// P2 items of slice s are issued L slices after its P1 items, so a P2 item only waits on
// items with smaller tickets, which are already held by running CTAs: no deadlock for any
// grid size, and Q is usually still in L2 when pass 2 re-reads it.
//
// Operand layouts (shared memory, 128-byte swizzle, 1024-byte aligned blocks of 64 columns):
//   Q, V, H tiles  [128 tokens][D]   K-major for S = Q U^T; MN-major (N = d) for A^T V
//   U              [MP anchors][D]   K-major
//   A tile         [128 tokens][128 anchors] MN-major as A^T (M = anchors) in pass 1,
//                  K-major as A (M = tokens) in pass 2; anchors >= MP stay zero
//   W' image       [D][MP]           K-major B operand of H = A W'
#include "common.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <math.h>

namespace anchor {

// Device-wide error word: bit 0 = an mbarrier wait timed out, bit 1 = a wait for another
// CTA's reduction timed out.  Read and cleared by anchor_attn_device_error().
__device__ unsigned int g_umma_error;

namespace {

using namespace ptx;

constexpr int kT = 128;                         // tokens per tile (UMMA M)
constexpr int kThreads = 128;                   // one thread per token row / TMEM lane
constexpr uint64_t kWaitNs = 2000000000ull;     // every wait gives up after 2 s

struct UParams {
    int slices, heads, n, m;
    float c;                  // scale * log2(e)
    int NT, C1, C2, L, total; // tiles per slice, P1 / P2 chunks per slice, lag, items
    float *part;              // [slices][C1][D][MP]  W partials (anchor index fastest)
    float *pdelta;            // [slices][C1][MP]     Delta partials
    uint16_t *wimg;           // [slices][D * MP]     W' operand images (bf16)
    unsigned *counts;         // [slices] finished P1 chunks
    unsigned *flags;          // [slices] W' ready
    unsigned *ticket;         // item counter
};

template <int D, int MP>
struct Layout {
    static constexpr int kQB = kT * D * 2;             // one Q / V / H tile
    static constexpr int kUB = MP * D * 2;
    static constexpr int kAB = kT * 128 * 2;           // A tile, 128 anchor columns
    static constexpr int kOnesB = 16 * kT * 2;         // 16 x 128 ones (bf16)
    static constexpr int kNS = 2;                      // TMA stages (each: a Q and a V tile)
    static constexpr int offU = 0;
    static constexpr int offQ = offU + kUB;            // kNS Q tiles
    static constexpr int offV = offQ + kNS * kQB;      // kNS V tiles; in pass 2: W' image, H staging
    static constexpr int offA = offV + kNS * kQB;
    static constexpr int offOnes = offA + kAB;
    static constexpr int offBar = offOnes + kOnesB;
    static constexpr int kBytes = offBar + 256;
    static constexpr int kSmem = kBytes + 1024;        // slack for 1024-byte alignment
    // TMEM columns: pass 1 uses S0 S1 W Delta, pass 2 uses S0 S1 H0 H1
    static constexpr int colS0 = 0, colS1 = MP, colW = 2 * MP, colD = 2 * MP + D;
    static constexpr int colH0 = 2 * MP, colH1 = 2 * MP + D;
    static constexpr int kColsNeeded = (2 * MP + D + 16) > (2 * MP + 2 * D) ? (2 * MP + D + 16) : (2 * MP + 2 * D);
    static constexpr int kTmemCols = kColsNeeded <= 256 ? 256 : 512;
    static_assert(kColsNeeded <= 512, "TMEM budget");
    static_assert(D * MP * 2 <= kQB, "W' image must fit in one V tile buffer");
    static_assert(offU % 1024 == 0 && offQ % 1024 == 0 && offV % 1024 == 0 && offA % 1024 == 0 &&
                  offOnes % 1024 == 0, "operand blocks must be 1024-byte aligned");
};

struct Item {
    int kind;   // 0 = P1, 1 = P2, 2 = FULL
    int slice;
    int chunk;
};

__device__ __forceinline__ Item decode(int t, const UParams &p) {
    if (p.C1 == 1) return {2, t, 0};
    const int S = p.slices, L = p.L, C1 = p.C1, C2 = p.C2;
    const int a = min(L, S);
    if (t < a * C1) return {0, t / C1, t % C1};
    t -= a * C1;
    if (L < S) {
        const int per = C1 + C2, nb = S - L;
        if (t < nb * per) {
            const int k = t / per, r = t - k * per;
            return r < C1 ? Item{0, L + k, r} : Item{1, k, r - C1};
        }
        t -= nb * per;
        return {1, (S - L) + t / C2, t % C2};
    }
    return {1, t / C2, t % C2};
}

// byte offset of 16-byte chunk `c` (0 .. cols/8-1) of row `r` in a swizzled [rows][cols]
// bf16 tile stored as 64-column blocks of `rows` x 128 bytes
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// byte offset of element (anchor j, column k) in the W' image [D rows][MP anchors]
template <int D>
__device__ __forceinline__ uint32_t wimg_off(int j, int k) {
    return (uint32_t)((j >> 6) * D * 128 + k * 128 + ((((j & 63) >> 3) ^ (k & 7)) << 4) + (j & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 2^x on the multi-function unit (PTX ex2.approx, flush-to-zero): one instruction.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Row softmax of one S row (TMEM lane = this thread's token), packed to bf16 pairs.
// Rows past the end of the slice become zero rows; anchors >= m get probability 0.
// The max and the sum run as 8 interleaved partial chains (fixed order: deterministic).
template <int MP>
__device__ __forceinline__ void softmax_row(uint32_t taddr_s, bool valid, int m, float c, uint32_t (&pk)[MP / 2]) {
    float v[MP];
#pragma unroll
    for (int q = 0; q < MP / 32; ++q) tmem_ld32(taddr_s + q * 32, v + q * 32);
    tmem_ld_wait();
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll
    for (int j = 0; j < MP; ++j) {
        v[j] *= c;
        if (j < m) mx8[j & 7] = fmaxf(mx8[j & 7], v[j]);
    }
    const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
    float z8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) z8[i] = 0.f;
#pragma unroll
    for (int j = 0; j < MP; ++j) {
        const float e = (j < m) ? ex2_approx(v[j] - mx) : 0.f;
        v[j] = e;
        z8[j & 7] += e;
    }
    const float z = ((z8[0] + z8[1]) + (z8[2] + z8[3])) + ((z8[4] + z8[5]) + (z8[6] + z8[7]));
    const float inv = valid ? 1.f / z : 0.f;
#pragma unroll
    for (int j = 0; j < MP / 2; ++j) pk[j] = pack_bf16x2(v[2 * j] * inv, v[2 * j + 1] * inv);
}

template <int MP>
__device__ __forceinline__ void store_a_row(const uint32_t (&pk)[MP / 2], uint8_t *sA, int row) {
#pragma unroll
    for (int c8 = 0; c8 < MP / 8; ++c8)
        *reinterpret_cast<uint4 *>(sA + sw_off(row, c8, kT)) =
            make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
}

template <int D, int MP>
__global__ void __launch_bounds__(kThreads, 1)
anchor_umma_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap th,
                   const UParams p) {
    using LY = Layout<D, MP>;
    constexpr int NS = LY::kNS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sU = sm + LY::offU;
    uint8_t *sQ = sm + LY::offQ;
    uint8_t *sV = sm + LY::offV;
    uint8_t *sA = sm + LY::offA;
    uint8_t *sOnes = sm + LY::offOnes;
    uint8_t *sW = sV;                 // pass 2: W' operand image (V buffer 0)
    uint8_t *sH = sV + LY::kQB;       // pass 2: H staging for the TMA store (V buffer 1)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::offBar);
    uint64_t *bar_q = bars;           // [NS] Q tile landed
    uint64_t *bar_v = bars + NS;      // [NS] V tile landed
    uint64_t *bar_u = bars + 2 * NS;  // U landed
    // MMA completion barriers; each has at most one phase in flight ahead of its waiters.
    uint64_t *bar_s = bars + 2 * NS + 1;  // [2] scores into S buffer 0 / 1 (and all MMAs before)
    uint64_t *bar_w = bars + 2 * NS + 3;  // A^T V + A^T 1 (pass 1) or A W' (pass 2)
    constexpr int kNumBars = 2 * NS + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kNumBars);
    int *s_item = reinterpret_cast<int *>(s_tmem + 1);
    int *s_last = s_item + 1;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid;  // token row of a tile / anchor row of W

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(bars + i, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tu);
        tma_prefetch_desc(&th);
    }
    for (int i = tid; i < LY::kOnesB / 4; i += kThreads) reinterpret_cast<uint32_t *>(sOnes)[i] = 0x3F803F80u;
    for (int i = tid; i < LY::kAB / 16; i += kThreads) reinterpret_cast<uint4 *>(sA)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 0) tmem_alloc(s_tmem, LY::kTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);

    const uint32_t sQa = smem_u32(sQ), sVa = smem_u32(sV), sUa = smem_u32(sU), sAa = smem_u32(sA);
    const uint32_t sOa = smem_u32(sOnes), sWa = smem_u32(sW);
    constexpr uint32_t kIdS = idesc_bf16_f32(128, MP, false, false);
    constexpr uint32_t kIdW = idesc_bf16_f32(128, D, true, true);
    constexpr uint32_t kIdD = idesc_bf16_f32(128, 16, true, false);
    constexpr uint32_t kIdH = idesc_bf16_f32(128, D, false, false);
    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_stream = policy_evict_first();

    // phases: TMA barriers are waited on by thread 0 only; MMA barriers by every thread
    uint32_t ph_q[NS], ph_v[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) ph_q[i] = ph_v[i] = 0u;
    uint32_t ph_u = 0u, ph_s[2] = {0u, 0u}, ph_w = 0u;
    bool ok = true;
    int cur_head = -1;

    auto wait = [&](uint64_t *bar, uint32_t &ph) {
        ok = mbar_wait(bar, ph, kWaitNs) && ok;
        ph ^= 1u;
    };
    // TMA of the Q / V tile `tile` of slice s into ring stage st.  Thread 0 only.  Tile k of
    // an item lives in stage (k - first tile) % NS of each ring; a stage is refilled once its
    // reader is done (Q: the score MMA, V: the A^T V MMA).
    auto load_q = [&](int s, int tile, int st) {
        mbar_arrive_expect_tx(bar_q + st, LY::kQB);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
            tma_load_3d(sQ + st * LY::kQB + b * kT * 128, &tq, bar_q + st, 64 * b, tile * kT, s, pol_keep);
    };
    auto load_v = [&](int s, int tile, int st) {
        mbar_arrive_expect_tx(bar_v + st, LY::kQB);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
            tma_load_3d(sV + st * LY::kQB + b * kT * 128, &tv, bar_v + st, 64 * b, tile * kT, s, pol_stream);
    };
    // Thread 0: wait for the Q tile in stage st, then S[buf] = Q U^T.
    auto issue_scores = [&](int st, int buf) {
        ok = mbar_wait(bar_q + st, ph_q[st], kWaitNs) && ok;
        ph_q[st] ^= 1u;
        tc_fence_after();
        const uint32_t dcol = buf ? LY::colS1 : LY::colS0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = smem_desc_sw128(sQa + st * LY::kQB + (kk >> 2) * kT * 128 + (kk & 3) * 32, 16, 1024);
            const uint64_t b = smem_desc_sw128(sUa + (kk >> 2) * MP * 128 + (kk & 3) * 32, 16, 1024);
            umma_bf16(tmem + dcol, a, b, kIdS, kk > 0);
        }
        umma_commit(bar_s + buf);
    };
    // All threads: H row of TMEM buffer `hcol` -> bf16 -> staging -> TMA store of tile `tile`.
    auto h_epilogue = [&](int s, int tile, uint32_t hcol) {
        uint32_t pk[D / 2];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            float v[32];
            tmem_ld32(trow + hcol + q * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[q * 16 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        }
        if (tid == 0) bulk_wait_group_read0();  // the previous store has read the staging buffer
        __syncthreads();
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8)
            *reinterpret_cast<uint4 *>(sH + sw_off(row, c8, kT)) =
                make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int bb = 0; bb < D / 64; ++bb)
                tma_store_3d(&th, sH + bb * kT * 128, 64 * bb, tile * kT, s, pol_stream);
            bulk_commit_group();
        }
    };

    for (;;) {
        if (tid == 0) *s_item = (int)atomicAdd(p.ticket, 1u);
        __syncthreads();
        const int t = *s_item;
        __syncthreads();
        if (t >= p.total) break;
        const Item it = decode(t, p);
        const int s = it.slice;
        const int h = s % p.heads;

        if (h != cur_head) {  // anchors of this head (all MMAs of the previous item are done)
            if (tid == 0) {
                mbar_arrive_expect_tx(bar_u, LY::kUB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b) tma_load_3d(sU + b * MP * 128, &tu, bar_u, 64 * b, 0, h, pol_keep);
            }
            wait(bar_u, ph_u);
            cur_head = h;
        }

        // ------------------------------------------------------------ pass 1
        if (it.kind != 1) {
            const int a = it.kind == 2 ? 0 : (int)((long long)it.chunk * p.NT / p.C1);
            const int b = it.kind == 2 ? p.NT : (int)((long long)(it.chunk + 1) * p.NT / p.C1);
            if (tid == 0) {
                for (int k = 0; k < NS && a + k < b; ++k) {
                    load_q(s, a + k, k);
                    load_v(s, a + k, k);
                }
                issue_scores(0, 0);
            }
            for (int tile = a; tile < b; ++tile) {
                const int i = tile - a, buf = i & 1, st = i % NS;
                wait(bar_s + buf, ph_s[buf]);          // S(tile) done: its Q stage is free
                tc_fence_after();
                if (tid == 0) {
                    if (tile + NS < b) load_q(s, tile + NS, st);
                    if (tile + 1 < b) issue_scores((i + 1) % NS, buf ^ 1);
                }
                uint32_t pk[MP / 2];
                softmax_row<MP>(trow + (buf ? LY::colS1 : LY::colS0), tile * kT + row < p.n, p.m, p.c, pk);
                if (i > 0) {
                    wait(bar_w, ph_w);                 // W(tile-1) done: A tile and V stage of tile-1 free
                    if (tid == 0 && tile - 1 + NS < b) load_v(s, tile - 1 + NS, (i - 1) % NS);
                }
                store_a_row<MP>(pk, sA, row);
                fence_proxy_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!ok)) goto abort;
                if (tid == 0) {
                    ok = mbar_wait(bar_v + st, ph_v[st], kWaitNs) && ok;
                    ph_v[st] ^= 1u;
                    tc_fence_after();
#pragma unroll
                    for (int kt = 0; kt < kT / 16; ++kt) {
                        const uint64_t ad = smem_desc_sw128(sAa + kt * 2048, 16384, 1024);
                        const uint64_t vd = smem_desc_sw128(sVa + st * LY::kQB + kt * 2048, 16384, 1024);
                        const uint64_t od = smem_desc_sw128(sOa + (kt >> 2) * 2048 + (kt & 3) * 32, 16, 1024);
                        const uint32_t acc = (tile > a || kt > 0) ? 1u : 0u;
                        umma_bf16(tmem + LY::colW, ad, vd, kIdW, acc);
                        umma_bf16(tmem + LY::colD, ad, od, kIdD, acc);
                    }
                    umma_commit(bar_w);
                }
            }
            wait(bar_w, ph_w);  // W, Delta of the chunk complete
            tc_fence_after();
            if (__syncthreads_or(!ok)) goto abort;

            if (it.kind == 0) {
                // chunk partial -> workspace; the last chunk of the slice reduces
                float v[32];
                float *dst = p.part + ((size_t)s * p.C1 + it.chunk) * (size_t)(D * MP);
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    tmem_ld32(trow + LY::colW + q * 32, v);
                    tmem_ld_wait();
                    if (row < MP) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) dst[(q * 32 + i) * MP + row] = v[i];
                    }
                }
                tmem_ld32(trow + LY::colD, v);
                tmem_ld_wait();
                if (row < MP) p.pdelta[((size_t)s * p.C1 + it.chunk) * MP + row] = v[0];
                __threadfence();
                tc_fence_before();
                __syncthreads();
                if (tid == 0) *s_last = (atomicAdd(p.counts + s, 1u) == (unsigned)(p.C1 - 1)) ? 1 : 0;
                __syncthreads();
                if (*s_last) {
                    __threadfence();
                    // Delta_j = sum over chunks in order; then W'_jk = W_jk / Delta_j
                    float *sd = reinterpret_cast<float *>(sA);  // A tile lower block is scratch now
                    if (tid < MP) {
                        float dsum = 0.f;
                        for (int cc = 0; cc < p.C1; ++cc) dsum += __ldcg(p.pdelta + ((size_t)s * p.C1 + cc) * MP + tid);
                        sd[tid] = dsum;
                    }
                    __syncthreads();
                    constexpr int JQ = MP / 4, KG = kThreads / JQ;
                    const int jq = tid % JQ, kg = tid / JQ;
                    const float *src = p.part + (size_t)s * p.C1 * (D * MP);
                    uint16_t *img = p.wimg + (size_t)s * (D * MP);
                    for (int k = kg; k < D; k += KG) {
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int cc = 0; cc < p.C1; ++cc) {
                            const float4 x = __ldcg(reinterpret_cast<const float4 *>(src + ((size_t)cc * D + k) * MP) + jq);
                            acc.x += x.x;
                            acc.y += x.y;
                            acc.z += x.z;
                            acc.w += x.w;
                        }
                        const float w4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * jq + e;
                            const float dj = sd[j];
                            const float wp = dj != 0.f ? w4[e] / dj : 0.f;
                            img[wimg_off<D>(j, k) / 2] = __bfloat16_as_ushort(__float2bfloat16_rn(wp));
                        }
                    }
                    __threadfence();
                    __syncthreads();
                    if (tid == 0) st_release_gpu(p.flags + s, 1u);
                    // the next softmax rewrites the lower block of the A tile
                }
                continue;
            }
            // FULL: W' = Delta^{-1} W straight from TMEM into the pass-2 operand image
            {
                float v[32], dj;
                tmem_ld32(trow + LY::colD, v);
                tmem_ld_wait();
                dj = v[0];
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    tmem_ld32(trow + LY::colW + q * 32, v);
                    tmem_ld_wait();
                    if (row < MP) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float wp = dj != 0.f ? v[i] / dj : 0.f;
                            *reinterpret_cast<uint16_t *>(sW + wimg_off<D>(row, q * 32 + i)) =
                                __bfloat16_as_ushort(__float2bfloat16_rn(wp));
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncthreads();
            }
        } else {
            // P2: wait for the slice's W' (published by another CTA), copy it on chip
            if (tid == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(p.flags + s) == 0u) {
                    if (globaltimer_ns() - t0 > kWaitNs) {
                        ok = false;
                        atomicOr(&g_umma_error, 2u);
                        break;
                    }
                    __nanosleep(128);
                }
            }
            if (__syncthreads_or(!ok)) goto abort;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.wimg + (size_t)s * (D * MP));
            for (int i = tid; i < D * MP * 2 / 16; i += kThreads)
                reinterpret_cast<uint4 *>(sW)[i] = __ldcg(src + i);
            fence_proxy_async_smem();
            __syncthreads();
        }

        // ------------------------------------------------------------ pass 2
        {
            const int a = it.kind == 2 ? 0 : (int)((long long)it.chunk * p.NT / p.C2);
            const int b = it.kind == 2 ? p.NT : (int)((long long)(it.chunk + 1) * p.NT / p.C2);
            if (tid == 0) {
                for (int k = 0; k < NS && a + k < b; ++k) load_q(s, a + k, k);
                issue_scores(0, 0);
            }
            for (int tile = a; tile < b; ++tile) {
                const int i = tile - a, buf = i & 1;
                wait(bar_s + buf, ph_s[buf]);          // S(tile) ready (and H(tile-1)'s inputs)
                tc_fence_after();
                if (tid == 0) {
                    if (tile + NS < b) load_q(s, tile + NS, i % NS);  // Q(tile) consumed
                    if (tile + 1 < b) issue_scores((i + 1) % NS, buf ^ 1);
                }
                uint32_t pk[MP / 2];
                softmax_row<MP>(trow + (buf ? LY::colS1 : LY::colS0), tile * kT + row < p.n, p.m, p.c, pk);
                if (i > 0) wait(bar_w, ph_w);          // H(tile-1) done: A tile free
                store_a_row<MP>(pk, sA, row);
                fence_proxy_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!ok)) goto abort;
                if (tid == 0) {
                    tc_fence_after();
                    const uint32_t hcol = buf ? LY::colH1 : LY::colH0;
#pragma unroll
                    for (int kj = 0; kj < MP / 16; ++kj) {
                        const uint64_t ad = smem_desc_sw128(sAa + (kj >> 2) * 16384 + (kj & 3) * 32, 16, 1024);
                        const uint64_t wd = smem_desc_sw128(sWa + (kj >> 2) * D * 128 + (kj & 3) * 32, 16, 1024);
                        umma_bf16(tmem + hcol, ad, wd, kIdH, kj > 0);
                    }
                    umma_commit(bar_w);
                }
                if (i > 0) {  // store H(tile-1) while the tensor core works on tile
                    tc_fence_after();
                    h_epilogue(s, tile - 1, buf ? LY::colH0 : LY::colH1);
                }
            }
            wait(bar_w, ph_w);
            tc_fence_after();
            if (__syncthreads_or(!ok)) goto abort;
            h_epilogue(s, b - 1, ((b - 1 - a) & 1) ? LY::colH1 : LY::colH0);
            tc_fence_before();
            if (tid == 0) bulk_wait_group_read0();
            __syncthreads();
        }
    }
    goto done;

abort:
    if (tid == 0) atomicOr(&g_umma_error, 1u);
done:
    if (tid == 0) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, LY::kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [outer][rows][cols] bf16 tensor, box = 64 columns x box_rows rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int cols, int rows, long long outer, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)outer};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * rows * 2};
    const cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int MP>
cudaError_t launch_t(const Problem &pr, const UmmaPlan &pl, void *ws, cudaStream_t stream) {
    using LY = Layout<D, MP>;
    auto kern = anchor_umma_kernel<D, MP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, LY::kSmem)) != cudaSuccess)
        return e;
    per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);

    CUtensorMap tq, tv, tu, th;
    const long long S = pr.slices();
    if (!make_map(&tq, pr.Q, D, pr.n, S, kT) || !make_map(&tv, pr.V, D, pr.n, S, kT) ||
        !make_map(&th, pr.H, D, pr.n, S, kT) || !make_map(&tu, pr.U, D, pr.m, pr.heads, MP))
        return cudaErrorInvalidValue;

    UParams p;
    p.slices = (int)S;
    p.heads = pr.heads;
    p.n = pr.n;
    p.m = pr.m;
    p.c = pr.scale * 1.4426950408889634f;
    p.NT = pl.NT;
    p.C1 = pl.C1;
    p.C2 = pl.C2;
    p.total = pl.total_items;
    const int grid = (int)std::min<long long>((long long)sms * per_sm, pl.total_items);
    p.L = pl.C1 == 1 ? 0 : std::max(1, std::min(p.slices, grid / (pl.C1 + pl.C2) + 2));
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.ticket = reinterpret_cast<unsigned *>(w);
    p.counts = reinterpret_cast<unsigned *>(w + 256);
    p.flags = p.counts + S;
    uint8_t *after = w + pl.header_bytes;
    p.pdelta = reinterpret_cast<float *>(after);
    p.part = p.pdelta + (size_t)S * pl.C1 * MP;
    p.wimg = reinterpret_cast<uint16_t *>(p.part + (size_t)S * pl.C1 * D * MP);
    if (pl.C1 == 1) p.part = p.pdelta = nullptr, p.wimg = nullptr;

    if ((e = cudaMemsetAsync(ws, 0, pl.header_bytes, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, LY::kSmem, stream>>>(tq, tv, tu, th, p);
    return cudaGetLastError();
}

}  // namespace

UmmaPlan umma_plan(const Problem &p) {
    UmmaPlan pl;
    const int MP = p.m <= 64 ? 64 : 128;
    pl.MP = MP;
    pl.NT = (p.n + kT - 1) / kT;
    const long long S = p.slices();
    pl.C1 = (pl.NT + kUmmaP1Tiles - 1) / kUmmaP1Tiles;
    if (pl.NT <= kUmmaFullTiles || pl.C1 == 1) {
        pl.C1 = 1;
        pl.C2 = 0;
        pl.total_items = (int)S;
        pl.header_bytes = 256;
        pl.workspace_bytes = 256;
        return pl;
    }
    pl.C2 = (pl.NT + kUmmaP2Tiles - 1) / kUmmaP2Tiles;
    pl.total_items = (int)(S * (pl.C1 + pl.C2));
    pl.header_bytes = (256 + 8 * (size_t)S + 1023) / 1024 * 1024;
    pl.workspace_bytes = pl.header_bytes + 4 * (size_t)S * pl.C1 * MP + 4 * (size_t)S * pl.C1 * p.d * MP +
                         2 * (size_t)S * p.d * MP;
    return pl;
}

bool umma_supported(const Problem &p) {
    return !p.f32 && (p.d == 64 || p.d == 128) && p.m >= 32 && p.m <= 128 &&
           p.slices() * ((p.n + kT - 1) / kT) * 3 < 0x7fffffffLL;
}

cudaError_t launch_umma(const Problem &p, const UmmaPlan &pl, void *workspace, cudaStream_t stream) {
    if (p.d == 64 && pl.MP == 64) return launch_t<64, 64>(p, pl, workspace, stream);
    if (p.d == 64 && pl.MP == 128) return launch_t<64, 128>(p, pl, workspace, stream);
    if (p.d == 128 && pl.MP == 64) return launch_t<128, 64>(p, pl, workspace, stream);
    if (p.d == 128 && pl.MP == 128) return launch_t<128, 128>(p, pl, workspace, stream);
    return cudaErrorInvalidValue;
}

cudaError_t umma_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_umma_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_umma_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

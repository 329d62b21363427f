// Tensor-core (tcgen05 / UMMA) variant of the anchor-attention forward
//   A = rowsoftmax(scale * Q U^T),  Delta = diag(colsum A),  H = A (Delta^{-1} (A^T V))
// (AnchorFormer, arXiv 2505.16463; pith.science verdict: "key_machinery", "core_discovery"
// and the referee summary of Eq. 11/12: B^T V -> Delta^{-1}(B^T V) -> B(Delta^{-1} B^T V)).
//
// One persistent kernel per call; work is cut into items that CTAs claim at run time:
//   P1(s, c)  pass 1 over token chunk c of slice s: per 128-token tile, S = Q U^T on the
//             tensor core (TMEM accumulator), row softmax in registers (one TMEM lane = one
//             token), A tile -> shared memory as bf16, then W += A^T V and Delta += A^T 1
//             on the tensor core (both from the same rounded A).  In plans that keep A for
//             pass 2 the A tile also goes to a workspace copy (TMA store, kept in L2).  The
//             chunk's (W, Delta) goes to a workspace partial; partials meet in a fixed binary
//             tree (the second of two siblings to arrive adds them: the sums do not depend on
//             which CTA ran what), and the root forms W' = Delta^{-1} W as a bf16 operand
//             image and publishes it.
//   P2(s, c)  pass 2 over token chunk c, once the slice's W' is published: A comes back
//             from the L2 copy, or (when every slice's copy would not fit L2) is recomputed
//             from Q into tensor memory; H = A W' on the tensor core, bf16 H rows to global
//             memory.  Stored A lines are dropped from L2 after use, without a write-back.
//   FULL(s)   short slices: P1 and P2 of a whole slice in one CTA, W' kept on chip; pass 2
//             recomputes A instead of storing it.
// A CTA takes a P2 chunk of a slice whose W' is ready, else a P1 chunk of a slice at most K
// slices past the oldest slice with unclaimed P2 chunks (K: the pass-2 operands of the slices
// in flight fit a share of L2; when all fit, every P1 chunk goes first).  A P2 chunk only
// waits on P1 chunks already held by running CTAs, so no grid size can deadlock.
//
// Roles (warp-specialised, one CTA per SM): warps 0-7 softmax (two groups of four), 8-11
// epilogue (H rows, partials, tree, W'), 12 TMA producer and work claiming, 13 issues
// S = Q U^T, 14 issues W, Delta and H.
//
// Operand layouts (shared memory, 128-byte swizzle, 1024-byte aligned blocks of 64 columns):
//   Q, V tiles     [128 tokens][D]   K-major for S = Q U^T; MN-major (N = d) for A^T V
//   U              [MP anchors][D]   K-major
//   A tile         [128 tokens][128 anchors] MN-major as A^T (M = anchors) for the W MMA;
//                  anchors >= MP stay zero.  MP = 64 with d = 64: only the 64 anchor columns,
//                  the W MMA's anchor rows 64..127 come from the ones block (never read back)
//   stored A       [128 tokens][MP]  K-major A operand of H = A W' (pass 2, ring slot)
//   W' image       [MP][D]           MN-major B operand of H = A W'
#include "common.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <math.h>

namespace anchor {

// Device-wide error word: bit 0 = a wait inside the kernel timed out, bit 1 = a wait for
// another CTA's reduction timed out.  Read and cleared by anchor_attn_device_error().
__device__ unsigned int g_umma_error;

namespace {

using namespace ptx;

constexpr int kT = 128;                         // tokens per tile (UMMA M)
// warps 0-7 softmax (two groups of four, each on half of the anchors of the same 128 rows),
// 8-11 epilogue, 12 producer, 13 issues S = Q U^T, 14 issues W, Delta and H
constexpr int kThreads = 480;
constexpr int kWarpProducer = 12, kWarpMmaS = 13, kWarpMmaX = 14;
constexpr int kIQ = 4;                          // item queue depth
constexpr uint64_t kWaitNs = 2000000000ull;     // a wait inside the CTA gives up after 2 s

struct UParams {
    int slices, heads, B, n, m;
    float c;                  // scale * log2(e)
    int NT, C1, C2;           // tiles per slice, P1 / P2 chunks per slice (C1 == 1: whole slices)
    int S2f, C2f;             // slices from schedule index S2f on cut pass 2 into C2f (finer) chunks
    float *part;              // [slices][C1][D/4][MP][4]  W partials (anchor-interleaved float4)
    float *pdelta;            // [slices][C1][MP]     Delta partials
    uint16_t *wimg;           // [slices][D * MP]     W' operand images (bf16, swizzled)
    uint16_t *abuf;           // [slices][n][MP]      A (bf16) written in pass 1, read in pass 2
    unsigned *flags;          // [slices * 32] W' published (one 128-byte line per slice)
    unsigned *p2c;            // [slices * 32] P2 chunks of the slice claimed so far
    unsigned *tree;           // [slices][C1] arrivals at the nodes of the reduction tree
    unsigned *next;           // next P1 chunk (or whole slice) to claim
    unsigned *head;           // first slice (schedule order) whose P2 chunks are not all claimed
    int K;                    // P1 may run at most K slices ahead of the P2 head
    int p1first;              // take every P1 chunk before any P2 chunk
    int store_a;              // pass 2 of split slices loads pass 1's A copy (else recomputes A)
    int hold_slice;           // failure-detection tests: this slice's W' is never published (-1: none)
    uint64_t wait_ns;         // limit of a wait on other CTAs (a slice's reduction)
};

template <int D, int MP>
struct Layout {
    static constexpr int kQB = kT * D * 2;             // one Q or V tile
    static constexpr int kATB = kT * MP * 2;           // one stored A tile (pass-2 operand)
    static constexpr int kSlotB = kQB > kATB ? kQB : kATB;  // ring slot: any of the three
    static constexpr int kUB = MP * D * 2;
    static constexpr int kWB = D * MP * 2;             // W' operand image
    // ones for Delta = A^T 1.  d = 64: a whole 128-token x 64-column MN-major block that the
    // W MMA reads as columns d .. d+15 of its B operand (W and Delta in one N = d + 16 MMA);
    // d = 128: a 16 x 128 K-major B operand of its own N = 16 MMA.
    static constexpr bool kFoldDelta = D == 64;
    // A tile: the W MMA is M = 128 (anchor rows).  With MP = 64 and the ones block at hand, the
    // tile holds only its 64 anchor columns and the MMA reads rows 64..127 from the ones block:
    // those rows of W and Delta are never read.  Otherwise 128 anchor columns.
    static constexpr bool kHalfA = MP == 64 && kFoldDelta;
    static constexpr int kAB = kT * (kHalfA ? 64 : 128) * 2;
    // softmax groups in ping-pong: with 64 anchors a thread holds a whole score row, so group
    // g takes the tiles of S buffer g whole (and A buffer g) instead of half of every row
    static constexpr bool kPP = kHalfA;
    static constexpr int kOnesB = kFoldDelta ? kT * 128 : 16 * kT * 2;
    static constexpr int kXchB = 2 * 2 * kT * 8;        // softmax halves' (max, sum), by tile parity
    static constexpr int kBarB = 1024;
    static constexpr int kMaxDyn = 227 * 1024 - 1024;  // minus the alignment slack
    // double-buffer the anchors and the A tile when that still leaves a 6-slot ring
    static constexpr bool kRoomy = (2 * kUB + 2 * kAB + 2 * kWB + kOnesB + kXchB + kBarB + 6 * kSlotB) <= kMaxDyn;
    static constexpr int kNU = kRoomy ? 2 : 1;
    static constexpr int kNA = kRoomy ? 2 : 1;
    static constexpr int kNW = kRoomy ? 2 : 1;
    // a single A buffer (pass 1 only): recomputed pass-2 H tiles are staged in the epilogue's
    // own buffer (4 KB per warp: 32 rows, one 64-column block at a time), so that their Q slot
    // goes back right after S and no pass-2 tile holds up the next pass-1 A tile; with two A
    // buffers there is no room for it, and H is staged in the Q slot
    static constexpr bool kStageH = kNA == 1;
    static constexpr int kHB = kStageH ? 4 * 32 * 128 : 0;
    // Single-buffered layouts can keep the pass-1 A tile and the pass-2 W' image in one buffer
    // (each pass uses only one of them) when that frees room for another ring slot; the two
    // uses then wait for each other's MMAs (barriers aw_w and aw_a below).
    static constexpr int kAWB = kAB > kWB ? kAB : kWB;
    static constexpr int kRest = kOnesB + kHB + kXchB + kBarB;
    static constexpr int kFixedSplit = kNU * kUB + kNA * kAB + kNW * kWB + kRest;
    static constexpr int kFixedUnion = kNU * kUB + kAWB + kRest;
    static constexpr bool kAW =
        kNA == 1 && kNW == 1 && (kMaxDyn - kFixedUnion) / kSlotB > (kMaxDyn - kFixedSplit) / kSlotB;
    static constexpr int kFixed = kAW ? kFixedUnion : kFixedSplit;
    static constexpr int kSlotsFit = (kMaxDyn - kFixed) / kSlotB;
    static constexpr int kNSlot = kSlotsFit > 8 ? 8 : kSlotsFit;
    // ring order per pass-1 tile: Q then V, or (a shallow ring) Q(t), then V(t-1), so that the
    // next S is not held up behind a V that is needed only after the softmax
    static constexpr bool kVLag = kNSlot < 5;
    static constexpr int offU = 0;
    static constexpr int offA = offU + kNU * kUB;
    static constexpr int offW = kAW ? offA : offA + kNA * kAB;
    static constexpr int offRing = kAW ? offA + kAWB : offW + kNW * kWB;
    static constexpr int offOnes = offRing + kNSlot * kSlotB;
    static constexpr int offH = offOnes + kOnesB;
    static constexpr int offXch = offH + kHB;
    static constexpr int offBar = offXch + kXchB;
    static constexpr int kBytes = offBar + kBarB;
    static constexpr int kSmem = kBytes + 1024;
    // TMEM: S0 | S1 | B0 (H0) | B1 (H1) and the pass-1 chunk accumulators W | Delta: two sets
    // of their own when they fit (a chunk starts while the epilogue drains the last one), else
    // one set over B0 | B1 (W at B0, Delta at B1 = B0 + D), shared with H
    static constexpr int colS0 = 0, colS1 = MP, colB0 = 2 * MP, colB1 = 2 * MP + D;
    static constexpr bool kWSep = 2 * MP + 2 * D + 2 * (D + 16) <= 512;
    static constexpr int colW0 = kWSep ? 2 * MP + 2 * D : colB0;
    static constexpr int colW1 = kWSep ? colW0 + D + 16 : colB0;
    static constexpr int kTmemCols = kWSep ? 512 : ((2 * MP + 2 * D) <= 256 ? 256 : 512);
    static_assert(kNSlot >= 3, "ring too shallow");
    static_assert(!kPP || (kNA == 2 && !kVLag), "ping-pong softmax: one A buffer per group, V right behind Q");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert(kUB % 1024 == 0 && offA % 1024 == 0 && offW % 1024 == 0 && offRing % 1024 == 0 &&
                  offOnes % 1024 == 0 && offH % 1024 == 0, "operand blocks must be 1024-byte aligned");
};

// Work items.  kind: 0 = P1 chunk, 1 = P2 chunk, 2 = whole slice, 3 = FLUSH (no tile follows
// soon: finish the tile held back for overlap), 4 = end of work.
struct Item {
    int kind;
    int slice;  // (batch, head) slice index b * heads + h
    int chunk;
};
constexpr int kFlush = 3, kEnd = 4;

// Slices are visited head-major (all batch entries of head 0, then head 1, ...) so that
// consecutive items usually share the anchors U.
__device__ __forceinline__ int slice_of(int so, const UParams &p) {
    const int h = so / p.B, b = so - h * p.B;
    return b * p.heads + h;
}

// One 128-token tile of an item, as every role sees it.
struct TileRef {
    int slice, tile;
    int kind;       // 0: pass-1 tile (S, softmax, A^T V);  1: pass-2 tile (S, softmax, A W')
    bool first;     // first tile of its pass within the item
    bool last;      // last tile of its pass within the item
    bool full;      // the item keeps W' on chip (whole slice per CTA)
    bool stored;    // pass-2 tile whose A is loaded from pass 1's copy instead of recomputed
    int chunk;      // pass-1 chunk (partials)
};

// P2 chunks of a slice: the last slices in schedule order take finer ones, so that the last
// round of pass-2 items spreads over every SM (the chunking of pass 2 does not change any sum)
__device__ __forceinline__ int c2_of(int slice, const UParams &p) {
    const int so = (slice % p.heads) * p.B + slice / p.heads;
    return so >= p.S2f ? p.C2f : p.C2;
}

__device__ __forceinline__ int item_tiles(const Item &it, const UParams &p, int &a1, int &b1) {
    if (it.kind == 2) {
        a1 = 0, b1 = p.NT;
        return 2 * p.NT;
    }
    const int C = it.kind == 0 ? p.C1 : c2_of(it.slice, p);
    a1 = (int)((long long)it.chunk * p.NT / C);
    b1 = (int)((long long)(it.chunk + 1) * p.NT / C);
    return b1 - a1;
}

__device__ __forceinline__ TileRef tile_at(const Item &it, int a1, int b1, int idx, const UParams &p) {
    TileRef r;
    r.slice = it.slice;
    r.chunk = it.chunk;
    r.full = it.kind == 2;
    r.stored = it.kind == 1 && p.store_a;
    const int n1 = b1 - a1;
    if (it.kind == 2) {
        const bool p2 = idx >= n1;
        const int k = p2 ? idx - n1 : idx;
        r.kind = p2 ? 1 : 0;
        r.tile = k;
        r.first = k == 0;
        r.last = k == n1 - 1;
    } else {
        r.kind = it.kind;
        r.tile = a1 + idx;
        r.first = idx == 0;
        r.last = idx == n1 - 1;
    }
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// byte offset of 16-byte chunk `c` (0 .. cols/8-1) of row `r` in a swizzled [rows][cols]
// bf16 tile stored as 64-column blocks of `rows` x 128 bytes
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The W' operand image holds W'[anchor j][column k] as MP rows of D bf16, in 64-column
// blocks of MP rows x 128 bytes, 128-byte swizzled (the layout a TMA load of a row-major
// [MP][D] tile produces): 8 consecutive columns of one anchor are one 16-byte chunk.
template <int MP>
__device__ __forceinline__ uint32_t wimg_chunk_off(int j, int c8) {
    return sw_off(j, c8, MP);
}

// 8 floats -> 8 bf16 (round to nearest even), scaled by r
__device__ __forceinline__ uint4 pack8_scaled(const float *x, float r) {
    return make_uint4(pack_bf16x2(x[0] * r, x[1] * r), pack_bf16x2(x[2] * r, x[3] * r),
                      pack_bf16x2(x[4] * r, x[5] * r), pack_bf16x2(x[6] * r, x[7] * r));
}


// 2^x on the multi-function unit (PTX ex2.approx, flush-to-zero): one instruction.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// named barriers of the two 4-warp groups (id 0 is __syncthreads)
__device__ __forceinline__ void sm_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void ep_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// one softmax group (ids 3, 4)
__device__ __forceinline__ void grp_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(3 + g) : "memory"); }

// Half of a row softmax: this thread's token row, anchors [col0, col0 + MP/2) of the S row.
// A_ij = softmax_j(scale * S_ij) = 2^(c S_ij - c max_j S_ij) / sum, c = scale * log2(e) > 0.
// The two halves of a row (two threads in the two softmax groups) each produce
//   e_j = 2^(c S_j - c mg)  with mg = their own maximum, and zg = sum of their e_j;
// the row then combines them: max M = max(mg0, mg1), sum z = zg0 2^(c(mg0 - M)) + zg1 2^(c(mg1 - M)),
// and A_j = e_j 2^(c(mg - M)) / z.  With MASKED, anchors >= m are -inf (probability 0).
// Max and sum run as 8 interleaved chains in a fixed order (deterministic).
template <int MP, bool MASKED>
__device__ __forceinline__ void softmax_half(uint32_t taddr, int col0, int m, float c, float (&v)[MP / 2], float &mg,
                                             float &zg) {
    constexpr int HM = MP / 2;
#pragma unroll
    for (int q = 0; q < HM / 32; ++q) tmem_ld32(taddr + q * 32, v + q * 32);
    tmem_ld_wait();
    if (MASKED) {
#pragma unroll
        for (int j = 0; j < HM; ++j)
            if (col0 + j >= m) v[j] = -INFINITY;
    }
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = v[i];
#pragma unroll
    for (int j = 8; j < HM; j += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            mx8[k] = (j + 8 + k < HM) ? max3_f32(mx8[k], v[j + k], v[j + 8 + k]) : fmaxf(mx8[k], v[j + k]);
    }
    mg = fmaxf(max3_f32(mx8[0], mx8[1], mx8[2]), max3_f32(max3_f32(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
    const float nb = mg == -INFINITY ? 0.f : -mg * c;  // a fully masked half: every e_j = 0
    const uint64_t c2 = f32x2(c, c), nb2 = f32x2(nb, nb);
    uint64_t z4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < HM; j += 2) {
        float a, b;
        f32x2_split(fma_f32x2(f32x2(v[j], v[j + 1]), c2, nb2), a, b);
        a = ex2_approx(a);
        b = ex2_approx(b);
        v[j] = a;
        v[j + 1] = b;
        z4[(j >> 1) & 3] = add_f32x2(z4[(j >> 1) & 3], f32x2(a, b));
    }
    float za, zb;
    f32x2_split(add_f32x2(add_f32x2(z4[0], z4[1]), add_f32x2(z4[2], z4[3])), za, zb);
    zg = za + zb;
}

template <int D, int MP>
__global__ void __launch_bounds__(kThreads, 1)
anchor_umma_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap ta_st,
                   const __grid_constant__ CUtensorMap ta_ld, const __grid_constant__ CUtensorMap th_st,
                   const UParams p, uint16_t *__restrict__ Hout) {
    using LY = Layout<D, MP>;
    constexpr int NS = LY::kNSlot, NU = LY::kNU, NA = LY::kNA, NW = LY::kNW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sU = sm + LY::offU;
    uint8_t *sA = sm + LY::offA;
    uint8_t *sW = sm + LY::offW;
    uint8_t *sRing = sm + LY::offRing;
    uint8_t *sOnes = sm + LY::offOnes;
    uint8_t *sH = sm + LY::offH;
    float2 *sXch = reinterpret_cast<float2 *>(sm + LY::offXch);  // [tile parity][group][row]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::offBar);
    // full/empty barrier pairs (arrival counts in brackets)
    uint64_t *slot_full = bars;                  // [NS] (1 + tx)  TMA landed
    uint64_t *slot_empty = slot_full + NS;       // [NS] (1)       MMA that read the slot completed
    uint64_t *s_full = slot_empty + NS;          // [2]  (1)       scores in S buffer
    uint64_t *s_empty = s_full + 2;              // [2]  (1)       S buffer free (read, or its P consumed)
    uint64_t *p_full = s_empty + 2;              // [2]  (1)       pass-2 A (P) written over the S buffer
    uint64_t *a_full = p_full + 2;               // [NA] (8, 4)    A tile written (one arrival per writing warp)
    uint64_t *a_empty = a_full + NA;             // [NA] (1)       MMA reading the A tile completed
    uint64_t *acc_full = a_empty + NA;           // [2]  (1)       W/Delta or H complete in TMEM
    uint64_t *acc_empty = acc_full + 2;          // [2]  (4)       epilogue read it
    uint64_t *wacc_full = acc_empty + 2;         // [2]  (1)       chunk W, Delta complete (separate sets)
    uint64_t *wacc_empty = wacc_full + 2;        // [2]  (4)       epilogue read them
    uint64_t *u_full = wacc_empty + 2;           // [NU] (1 + tx)  U landed
    uint64_t *u_empty = u_full + NU;             // [NU] (1)       MMAs on that U completed
    uint64_t *w_full = u_empty + NU;             // [NW] (1 [+ tx]) W' image in place
    uint64_t *w_empty = w_full + NW;             // [NW] (1)       MMAs reading W' completed
    uint64_t *iq_full = w_empty + NW;            // [kIQ] (1)      item queue
    uint64_t *iq_empty = iq_full + kIQ;          // [kIQ] (4)
    uint64_t *mma_done = iq_empty + kIQ;         // [2]  (1)       every MMA of an issuer completed (exit)
    // one A / W' buffer (LY::kAW): the MMAs before a W' load, or before a pass-1 A tile that
    // follows a pass-2 phase, have completed (committed by the W/H issuer at those points)
    uint64_t *aw_w = mma_done + 2;               // (1)
    uint64_t *aw_a = aw_w + 1;                   // (1)
    constexpr int kNumBars = 2 * NS + 2 + 2 + 2 + 2 * NA + 2 + 2 + 2 + 2 + 2 * NU + 2 * NW + 2 * kIQ + 2 + 2;
    static_assert(kNumBars * 8 + 3 * 4 * kIQ + 16 + 4 * NS <= LY::kBarB, "barrier area");
    int *s_items = reinterpret_cast<int *>(bars + kNumBars);           // [kIQ][3]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_items + 3 * kIQ);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_last = reinterpret_cast<int *>(s_tmem + 2);
    uint32_t *s_ast = s_tmem + 3;  // softmax-warp chunk ends whose A stores are complete
    // ring slot tags: the load sequence number a slot was last filled with.  Two threads
    // consume the ring, each skipping the other's slots, so a parity wait alone could match a
    // phase two loads old; a consumer first sees its own tag, then waits for the phase.
    uint32_t *s_slot_seq = s_tmem + 4;  // [NS]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(slot_full + i, 1);
            mbar_init(slot_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(s_empty + i, 1);
            mbar_init(p_full + i, 1);
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, 4);
            mbar_init(wacc_full + i, 1);
            mbar_init(wacc_empty + i, 4);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(a_full + i, LY::kPP ? 4 : 8);
            mbar_init(a_empty + i, 1);
        }
        for (int i = 0; i < NU; ++i) {
            mbar_init(u_full + i, 1);
            mbar_init(u_empty + i, 1);
        }
        for (int i = 0; i < NW; ++i) {
            mbar_init(w_full + i, 1);
            mbar_init(w_empty + i, 1);
        }
        for (int i = 0; i < kIQ; ++i) {
            mbar_init(iq_full + i, 1);
            mbar_init(iq_empty + i, 4);
        }
        mbar_init(mma_done + 0, 1);
        mbar_init(mma_done + 1, 1);
        mbar_init(aw_w, 1);
        mbar_init(aw_a, 1);
        *s_abort = 0;
        *s_ast = 0;
        for (int i = 0; i < NS; ++i) s_slot_seq[i] = 0xffffffffu;
        fence_mbar_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tu);
        tma_prefetch_desc(&ta_st);
        tma_prefetch_desc(&ta_ld);
        tma_prefetch_desc(&th_st);
    }
    for (int i = tid; i < LY::kOnesB / 4; i += kThreads) reinterpret_cast<uint32_t *>(sOnes)[i] = 0x3F803F80u;
    for (int i = tid; i < NA * LY::kAB / 16; i += kThreads) reinterpret_cast<uint4 *>(sA)[i] = make_uint4(0, 0, 0, 0);
    if (warp == kWarpMmaS) tmem_alloc(s_tmem, LY::kTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // Bounded wait that also gives up once another role has given up.
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
            if (*s_abort) return false;
            if (globaltimer_ns() - t0 > kWaitNs) {
                *s_abort = 1;
                atomicOr(&g_umma_error, 1u);
                return false;
            }
        }
    };
    // Bounded wait on the way out, after a wait gave up: it ignores the abort flag, because
    // it lets copies and MMAs that were already issued finish before the CTA leaves.
    auto drain_wait = [&](uint64_t *bar, uint32_t parity) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (globaltimer_ns() - t0 > kWaitNs) {
                atomicOr(&g_umma_error, 4u);
                return;
            }
            __nanosleep(128);
        }
    };
    // wait for ring load number `seq` (see s_slot_seq)
    auto wait_slot = [&](uint32_t seq) -> bool {
        uint32_t *tag = s_slot_seq + seq % NS;
        if (ld_acquire_cta(tag) != seq) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_cta(tag) != seq) {
                if (*s_abort) return false;
                if (globaltimer_ns() - t0 > kWaitNs) {
                    *s_abort = 1;
                    atomicOr(&g_umma_error, 1u);
                    return false;
                }
                __nanosleep(32);
            }
        }
        return wait(slot_full + seq % NS, (seq / NS) & 1u);
    };
    auto read_item = [&](uint32_t iq) -> Item {
        const int *e = s_items + 3 * (int)(iq % kIQ);
        return {e[0], e[1], e[2]};
    };

    if (warp == kWarpProducer) {
        // =========================================================== producer (whole warp:
        // every lane waits and decides alike; lane 0 issues the copies and the queue writes)
        constexpr unsigned FULLW = 0xffffffffu;
        const bool L0 = lane == 0;
        const uint64_t pol_keep = policy_evict_last();
        const uint64_t pol_stream = policy_evict_first();
        uint32_t ld_seq = 0, iq = 0, wuse = 0, nu = 0, nww = 0;  // nww: W' loads (aw_w phases)
        uint32_t wl_use[2] = {0u, 0u};  // per W' buffer: 1 + the use its last load was for (0: none)
        int u_head = -1;
        TileRef pend_v;
        bool has_pend_v = false, ok = true, flushed = true;
        const unsigned S = (unsigned)p.slices;
        const unsigned n1 = (unsigned)(p.C1 == 1 ? p.slices : p.slices * p.C1);
        const unsigned n2 = (unsigned)(p.C1 == 1 ? 0 : p.slices * p.C2);
        auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(FULLW, wait(bar, parity)) != 0;
        };
        // one 128-row tile of `cols` columns (D for Q and V, MP for a stored A tile)
        auto load_slot = [&](const CUtensorMap *map, int slice, int tile, uint64_t pol, int cols) -> bool {
            const int st = (int)(ld_seq % NS);
            if (!wwait(slot_empty + st, ((ld_seq / NS) & 1u) ^ 1u)) return false;
            if (L0) {
                st_release_cta(s_slot_seq + st, ld_seq);
                mbar_arrive_expect_tx(slot_full + st, (uint32_t)(kT * cols * 2));
                for (int b = 0; b < cols / 64; ++b)
                    tma_load_3d(sRing + st * LY::kSlotB + b * kT * 128, map, slot_full + st, 64 * b, tile * kT, slice, pol);
            }
            ++ld_seq;
            return true;
        };
        auto push = [&](const Item &it) -> bool {
            const int qs = (int)(iq % kIQ);
            if (!wwait(iq_empty + qs, ((iq / kIQ) & 1u) ^ 1u)) return false;
            if (L0) {
                s_items[3 * qs] = it.kind;
                s_items[3 * qs + 1] = it.slice;
                s_items[3 * qs + 2] = it.chunk;
                mbar_arrive(iq_full + qs);
            }
            ++iq;
            return true;
        };
        auto vload = [](const unsigned *a) { return *reinterpret_cast<const volatile unsigned *>(a); };
        // Claim the next item: a P2 chunk of a slice whose W' is published (the 32 lanes test
        // 32 slices from the head at once, with plain loads), else a P1 chunk if its slice is
        // within K of the head, or a whole slice.  Every atomic is an add or a max: no
        // compare-and-swap retries.  1: claimed, 0: nothing claimable yet, -1: no work left.
        auto claim = [&](Item &it) -> int {
            int r = 0;
            unsigned u = 0;
            if (n2 == 0) {
                if (L0) {
                    if (vload(p.next) >= n1) {
                        r = -1;
                    } else {
                        u = atomicAdd(p.next, 1u);
                        r = u < n1 ? 1 : -1;
                    }
                }
                r = __shfl_sync(FULLW, r, 0);
                u = __shfl_sync(FULLW, u, 0);
                if (r == 1) it = {2, slice_of((int)u, p), 0};
                return r;
            }
            auto try_p1 = [&](unsigned limit) -> bool {  // P1 chunk whose slice is below `limit`
                int got = 0;
                unsigned v = 0;
                if (L0) {
                    const unsigned nx = vload(p.next);
                    if (nx < n1 && nx / (unsigned)p.C1 < limit) {
                        v = atomicAdd(p.next, 1u);
                        got = v < n1 ? 1 : 0;
                    }
                }
                got = __shfl_sync(FULLW, got, 0);
                v = __shfl_sync(FULLW, v, 0);
                if (got) {
                    const int so = (int)(v / (unsigned)p.C1);
                    it = {0, slice_of(so, p), (int)(v - (unsigned)so * p.C1)};
                }
                return got != 0;
            };
            if (p.p1first && try_p1(S)) return 1;
            unsigned h = __shfl_sync(FULLW, L0 ? vload(p.head) : 0u, 0);
            for (;;) {
                if (h >= S) return -1;
                const unsigned so = h + (unsigned)lane;
                bool exhausted = true, ready = false;
                int sl = 0;
                if (so < S) {
                    sl = slice_of((int)so, p);
                    exhausted = vload(p.p2c + 32 * sl) >= (unsigned)c2_of(sl, p);
                    ready = !exhausted && vload(p.flags + 32 * sl) != 0u;
                }
                const unsigned ex = __ballot_sync(FULLW, exhausted);
                if (ex == FULLW) {  // all 32 exhausted: move the head on
                    h = min(h + 32u, S);
                    if (L0) atomicMax(p.head, h);
                    continue;
                }
                const unsigned nh = h + (unsigned)(__ffs(~ex) - 1);
                if (nh > h && L0) atomicMax(p.head, nh);
                h = nh;
                // ready slices of the head whose U is already in shared memory go first
                const unsigned rs = __ballot_sync(FULLW, ready && sl % p.heads == u_head);
                const unsigned rm = __ballot_sync(FULLW, ready);
                for (unsigned pass = 0; pass < 2; ++pass) {
                    unsigned rq = pass == 0 ? rs : rm & ~rs;
                    while (rq) {
                        const int ln = __ffs(rq) - 1;
                        unsigned got = 0;
                        if (lane == ln) got = atomicAdd(p.p2c + 32 * sl, 1u);
                        got = __shfl_sync(FULLW, got, ln);
                        const int slr = __shfl_sync(FULLW, sl, ln);
                        if (got < (unsigned)c2_of(slr, p)) {
                            it = {1, slr, (int)got};
                            return 1;
                        }
                        rq &= rq - 1u;
                    }
                }
                break;
            }
            if (!p.p1first && try_p1(h + (unsigned)p.K)) return 1;
            return 0;
        };
        uint64_t idle_since = 0;
        uint32_t backoff = 256;
        bool idle = false;
        Item ahead;
        bool have_ahead = false;
        while (ok) {
            Item it;
            int r;
            if (have_ahead) {
                it = ahead;
                have_ahead = false;
                r = 1;
            } else {
                r = claim(it);
            }
            if (r == 0) {  // the remaining P2 chunks wait for reductions still running
                if (!idle) {
                    idle = true;
                    idle_since = globaltimer_ns();
                }
                if (!flushed) {
                    ok = push(Item{kFlush, 0, 0});
                    if (ok && has_pend_v) ok = load_slot(&tv, pend_v.slice, pend_v.tile, pol_stream, D);
                    has_pend_v = false;
                    flushed = true;
                }
                const bool give_up = __any_sync(FULLW, *s_abort != 0 || globaltimer_ns() - idle_since > p.wait_ns);
                if (give_up) {
                    if (L0 && !*s_abort) {
                        *s_abort = 1;
                        atomicOr(&g_umma_error, 2u);
                    }
                    break;
                }
                __nanosleep(backoff);
                backoff = backoff < 1024 ? 2 * backoff : 1024;
                continue;
            }
            backoff = 256;
            idle = false;
            if (r < 0) {
                ok = push(Item{kEnd, 0, 0});
                break;
            }
            if (!push(it)) break;
            flushed = false;
            const int h = it.slice % p.heads;
            // U load number nu goes to buffer nu % NU (pass 2 on a stored A needs no U)
            if ((it.kind != 1 || !p.store_a) && h != u_head) {
                const int ub = (int)(nu % NU);
                if (!wwait(u_empty + ub, ((nu / NU) & 1u) ^ 1u)) break;
                if (L0) {
                    mbar_arrive_expect_tx(u_full + ub, LY::kUB);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(sU + ub * LY::kUB + b * MP * 128, &tu, u_full + ub, 64 * b, 0, h, pol_keep);
                }
                u_head = h;
                ++nu;
            }
            int a1, b1;
            const int nt = item_tiles(it, p, a1, b1);
            for (int idx = 0; idx < nt && ok; ++idx) {
                const TileRef tr = tile_at(it, a1, b1, idx, p);
                // Q is kept in L2 only for a whole-slice item, whose pass 2 follows at once: across
                // split slices too much streams through L2 before pass 2 comes back to it
                if (tr.stored) ok = load_slot(&ta_ld, tr.slice, tr.tile, pol_stream, MP);
                else ok = load_slot(&tq, tr.slice, tr.tile, tr.kind == 0 && tr.full ? pol_keep : pol_stream, D);
                if (ok && has_pend_v) {
                    ok = load_slot(&tv, pend_v.slice, pend_v.tile, pol_stream, D);
                    has_pend_v = false;
                }
                if (tr.kind == 0) {
                    if (LY::kVLag) {
                        pend_v = tr;
                        has_pend_v = true;
                    } else if (ok) {
                        ok = load_slot(&tv, tr.slice, tr.tile, pol_stream, D);
                    }
                }
                if (ok && tr.kind == 1 && tr.first) {
                    if (!tr.full) {  // W' of a split slice: published (claim checked the flag)
                        const int wb = (int)(wuse % NW);
                        ok = wwait(w_empty + wb, ((wuse / NW) & 1u) ^ 1u);
                        // one A / W' buffer: the last pass-1 tile's MMAs have read its A
                        if (LY::kAW) ok = ok && wwait(aw_w, nww & 1u);
                        ++nww;
                        if (ok && L0) {
                            (void)ld_acquire_gpu(p.flags + 32 * tr.slice);  // orders the image reads
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                            mbar_arrive_expect_tx(w_full + wb, LY::kWB);
                            bulk_load(sW + wb * LY::kWB, p.wimg + (size_t)tr.slice * (D * MP), LY::kWB, w_full + wb);
                            wl_use[wb] = wuse + 1u;
                        }
                    }
                    ++wuse;
                }
                // claim the next item once this one's loads are all issued, so that the claim's
                // memory round trips overlap the consumers working through the full ring; a
                // whole-slice item is a few tiles long, and claims after its first
                if (ok && idx == (it.kind == 2 ? 0 : nt - 1) && !have_ahead) have_ahead = claim(ahead) == 1;
            }
        }
        if (ok && has_pend_v) load_slot(&tv, pend_v.slice, pend_v.tile, pol_stream, D);
        // Leave no copy in flight: after a wait gave up, loads may still be landing in the
        // ring, U and W' buffers.  Each buffer's newest load completes its own phase.
        for (uint32_t q = ld_seq > (uint32_t)NS ? ld_seq - NS : 0u; q < ld_seq; ++q)
            drain_wait(slot_full + q % NS, (q / NS) & 1u);
        for (uint32_t q = nu > (uint32_t)NU ? nu - NU : 0u; q < nu; ++q) drain_wait(u_full + q % NU, (q / NU) & 1u);
        for (int b = 0; b < NW; ++b)
            if (wl_use[b]) drain_wait(w_full + b, ((wl_use[b] - 1u) / NW) & 1u);
    } else if (warp == kWarpMmaS || warp == kWarpMmaX) {
        // =========================================================== MMA issue
        // Two issuing threads, so that neither kind of MMA waits behind the other: warp 13
        // issues S = Q U^T as soon as a Q tile and an S buffer are there; warp 14 issues
        // W += A^T V, Delta += A^T 1 and H = A W' as soon as their A tile is written.  Both
        // replay the producer's ring order from the item stream: per tile one slot (Q, or a
        // stored A), then the previous pass-1 tile's V.  Descriptors advance by adding the
        // K-step offset to the start-address field.
        if (lane == 0) {
            const uint32_t sRa = smem_u32(sRing);
            uint32_t lseq = 0, iq = 0;
            bool lpend = false, ok = true;
            if (warp == kWarpMmaS) {
                constexpr uint32_t kIdS = idesc_bf16_f32(128, MP, false, false);
                const uint32_t sUa = smem_u32(sU);
                uint32_t sidx = 0, nu = 0;
                int prev_head = -1;
                while (ok) {
                    if (!wait(iq_full + iq % kIQ, (iq / kIQ) & 1u)) break;
                    const Item it = read_item(iq);
                    mbar_arrive(iq_empty + iq % kIQ);
                    ++iq;
                    if (it.kind == kEnd) break;
                    if (it.kind == kFlush) {
                        if (lpend) ++lseq;
                        lpend = false;
                        continue;
                    }
                    const int h = it.slice % p.heads;
                    if ((it.kind != 1 || !p.store_a) && h != prev_head) {
                        if (prev_head >= 0) umma_commit(u_empty + (nu - 1) % NU);  // every S on the old U issued
                        if (!wait(u_full + nu % NU, (nu / NU) & 1u)) break;
                        ++nu;
                        prev_head = h;
                    }
                    const uint64_t bdesc = smem_desc_sw128(sUa + ((nu - 1) % NU) * LY::kUB, 16, 1024);
                    int a1, b1;
                    const int nt = item_tiles(it, p, a1, b1);
                    for (int idx = 0; idx < nt && ok; ++idx) {
                        const TileRef tr = tile_at(it, a1, b1, idx, p);
                        const uint32_t mseq = lseq++;
                        if (LY::kVLag) {
                            if (lpend) ++lseq;
                            lpend = tr.kind == 0;
                        } else if (tr.kind == 0) {
                            ++lseq;  // this tile's V
                        }
                        if (tr.stored) continue;
                        const int qslot = (int)(mseq % NS);
                        if (!wait_slot(mseq)) { ok = false; break; }
                        const int sb = (int)(sidx & 1u);
                        if (!wait(s_empty + sb, ((sidx >> 1) & 1u) ^ 1u)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t dcol = sb ? LY::colS1 : LY::colS0;
                        const uint64_t adesc = smem_desc_sw128(sRa + qslot * LY::kSlotB, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            umma_bf16(tmem + dcol, adesc + (uint64_t)((((kk >> 2) * kT * 128) + (kk & 3) * 32) >> 4),
                                      bdesc + (uint64_t)((((kk >> 2) * MP * 128) + (kk & 3) * 32) >> 4), kIdS, kk > 0);
                        umma_commit(s_full + sb);
                        // unless the epilogue has a staging buffer of its own, a pass-2 tile's Q slot
                        // stays held: the epilogue stages the H tile there
                        if (tr.kind == 0 || LY::kStageH) umma_commit(slot_empty + qslot);
                        ++sidx;
                    }
                }
            } else {
                constexpr uint32_t kIdW = idesc_bf16_f32(128, D, true, true);
                constexpr uint32_t kIdD = idesc_bf16_f32(128, 16, true, false);
                constexpr uint32_t kIdWD = idesc_bf16_f32(128, D + 16, true, true);  // W | Delta
                const uint32_t sOnesA = smem_u32(sOnes);
                constexpr uint32_t kIdH = idesc_bf16_f32(128, D, false, true);
                const uint32_t sAa = smem_u32(sA), sWa = smem_u32(sW);
                const uint64_t odesc = smem_desc_sw128(smem_u32(sOnes), 16, 1024);
                uint32_t xk = 0, wuse = 0, p2 = 0;
                uint32_t accuse[2] = {0u, 0u};
                TileRef pv;
                int pvs = 0;  // its S buffer
                uint32_t xs = 0, pcnt[2] = {0u, 0u};  // S tiles seen; pass-2 A's seen per S buffer
                uint32_t acnt[2] = {0u, 0u};          // ping-pong: pass-1 A's seen per A buffer
                uint32_t xw = 0;                      // pass-1 chunks started (separate W sets)
                bool after_p2 = false;                // a pass-2 tile since the last pass-1 tile
                // H = A W' into the next H buffer; A at `adesc` (K-major, shared memory) or, with
                // from_tmem, in tensor memory at a_tmem
                auto issue_h = [&](const TileRef &tr, uint64_t adesc, uint32_t a_tmem, bool from_tmem) -> bool {
                    const int wb = (int)((tr.first ? wuse : wuse - 1u) % NW);  // this pass-2 phase's W'
                    if (tr.first) {
                        if (LY::kAW && !tr.full) umma_commit(aw_w);  // the producer may load W' over A
                        if (!wait(w_full + wb, (wuse / NW) & 1u)) return false;
                        ++wuse;
                    }
                    const int hb = (int)(p2 & 1u);
                    if (!wait(acc_empty + hb, (accuse[hb] & 1u) ^ 1u)) return false;
                    tc_fence_after();
                    const uint64_t wdesc = smem_desc_sw128(sWa + wb * LY::kWB, MP * 128, 1024);
                    const uint32_t dcol = hb ? LY::colB1 : LY::colB0;
                    if (from_tmem) {
#pragma unroll
                        for (int kj = 0; kj < MP / 16; ++kj)
                            umma_bf16_tmem_a(tmem + dcol, a_tmem + kj * 8, wdesc + (uint64_t)(kj * 128), kIdH, kj > 0);
                    } else {
#pragma unroll
                        for (int kj = 0; kj < MP / 16; ++kj)
                            umma_bf16(tmem + dcol, adesc + (uint64_t)((((kj >> 2) * kT * 128) + (kj & 3) * 32) >> 4),
                                      wdesc + (uint64_t)(kj * 128), kIdH, kj > 0);
                    }
                    umma_commit(acc_full + hb);
                    ++accuse[hb];
                    ++p2;
                    if (tr.last) umma_commit(w_empty + wb);
                    return true;
                };
                // pass 1: W += A^T V, Delta += A^T 1 from the softmax's A tile (V at ring position vseq)
                // (sbx: the tile's S buffer, which names its A buffer in ping-pong)
                auto do_x = [&](const TileRef &tr, uint32_t vseq, int sbx) -> bool {
                    const int ab = LY::kPP ? sbx : (int)(xk % NA);
                    if (!wait(a_full + ab, LY::kPP ? (acnt[sbx] & 1u) : ((xk / NA) & 1u))) return false;
                    if (LY::kPP) ++acnt[sbx];
                    const uint32_t sAb = sAa + ab * LY::kAB;
                    if (tr.kind == 0) {
                        const int vs = (int)(vseq % NS);
                        if (!wait_slot(vseq)) return false;
                        const int wbuf = (int)(xw & 1u);
                        if (tr.first) {
                            if constexpr (LY::kWSep) {
                                if (!wait(wacc_empty + wbuf, ((xw >> 1) & 1u) ^ 1u)) return false;
                            } else {
                                if (!wait(acc_empty + 0, (accuse[0] & 1u) ^ 1u)) return false;
                                if (!wait(acc_empty + 1, (accuse[1] & 1u) ^ 1u)) return false;
                            }
                        }
                        const uint32_t wcol = wbuf ? LY::colW1 : LY::colW0;
                        tc_fence_after();
                        // second 64-anchor block of A^T: the tile's own, or the ones block
                        const uint64_t adesc = smem_desc_sw128(sAb, LY::kHalfA ? sOnesA - sAb : 16384, 1024);
                        if constexpr (LY::kFoldDelta) {
                            // second 64-column block of B = the ones block: the leading-byte
                            // offset spans from this slot to it (columns D.. of the result =
                            // Delta)
                            const uint32_t vbase = sRa + vs * LY::kSlotB;
                            const uint64_t vdesc = smem_desc_sw128(vbase, sOnesA - vbase, 1024);
#pragma unroll
                            for (int kt = 0; kt < kT / 16; ++kt)
                                umma_bf16(tmem + wcol, adesc + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), kIdWD,
                                          (!tr.first || kt > 0) ? 1u : 0u);
                        } else {
                            const uint64_t vdesc = smem_desc_sw128(sRa + vs * LY::kSlotB, 16384, 1024);
#pragma unroll
                            for (int kt = 0; kt < kT / 16; ++kt) {
                                const uint32_t acc = (!tr.first || kt > 0) ? 1u : 0u;
                                umma_bf16(tmem + wcol, adesc + (uint64_t)(kt * 128), vdesc + (uint64_t)(kt * 128), kIdW, acc);
                                umma_bf16(tmem + wcol + D, adesc + (uint64_t)(kt * 128),
                                          odesc + (uint64_t)((((kt >> 2) * 2048) + (kt & 3) * 32) >> 4), kIdD, acc);
                            }
                        }
                        umma_commit(a_empty + ab);
                        umma_commit(slot_empty + vs);
                        if (tr.last) {
                            if constexpr (LY::kWSep) {
                                umma_commit(wacc_full + wbuf);
                            } else {
                                umma_commit(acc_full + 0);
                                umma_commit(acc_full + 1);
                                ++accuse[0];
                                ++accuse[1];
                            }
                            ++xw;
                        }
                    }
                    ++xk;
                    return true;
                };
                while (ok) {
                    if (!wait(iq_full + iq % kIQ, (iq / kIQ) & 1u)) break;
                    const Item it = read_item(iq);
                    mbar_arrive(iq_empty + iq % kIQ);
                    ++iq;
                    if (it.kind == kEnd) break;
                    if (it.kind == kFlush) {  // the producer loads the held-back V now
                        if (lpend && !do_x(pv, lseq++, pvs)) break;
                        lpend = false;
                        continue;
                    }
                    int a1, b1;
                    const int nt = item_tiles(it, p, a1, b1);
                    for (int idx = 0; idx < nt && ok; ++idx) {
                        const TileRef tr = tile_at(it, a1, b1, idx, p);
                        if (LY::kAW) {  // one A / W' buffer: the softmax may write A once W' is read
                            if (tr.kind == 0 && after_p2) umma_commit(aw_a);
                            after_p2 = tr.kind == 1;
                        }
                        const uint32_t mseq = lseq++;
                        if (lpend) {  // the previous pass-1 tile's V follows this tile's first slot
                            if (!do_x(pv, lseq++, pvs)) { ok = false; break; }
                            lpend = false;
                        }
                        const int sbx = (int)(xs & 1u);  // this tile's S buffer (tiles with an S only)
                        if (!tr.stored) ++xs;
                        if (tr.kind == 0) {
                            if (LY::kVLag) {
                                pv = tr;
                                pvs = sbx;
                                lpend = true;
                            } else if (!do_x(tr, lseq++, sbx)) {  // its V is right behind its Q
                                ok = false;
                                break;
                            }
                        } else if (tr.stored) {
                            // the slot holds the A tile pass 1 stored; the epilogue releases it
                            const int aslot = (int)(mseq % NS);
                            if (!wait_slot(mseq)) { ok = false; break; }
                            if (!issue_h(tr, smem_desc_sw128(sRa + aslot * LY::kSlotB, 16, 1024), 0u, false)) { ok = false; break; }
                        } else {
                            // recomputed pass-2 A, written by the softmax over its S buffer
                            if (!wait(p_full + sbx, pcnt[sbx] & 1u)) { ok = false; break; }
                            ++pcnt[sbx];
                            if (!issue_h(tr, 0ull, tmem + (sbx ? LY::colS1 : LY::colS0), true)) { ok = false; break; }
                            umma_commit(s_empty + sbx);
                        }
                    }
                }
                if (ok && lpend) do_x(pv, lseq++, pvs);  // after the end marker the producer loads the last V
            }
            // every MMA this thread issued has completed before the CTA leaves (after a wait
            // gave up, nothing else waits for them)
            umma_commit(mma_done + (warp - kWarpMmaS));
            drain_wait(mma_done + (warp - kWarpMmaS), 0u);
        }
    } else if (warp < 8) {
        // =========================================================== softmax (warps 0-7)
        // Group g = warp / 4 takes anchors [g MP/2, (g+1) MP/2) of the rows of TMEM lane
        // quadrant warp % 4; the two halves of a row meet through shared memory.
        const int g = warp >> 2, quad = warp & 3;
        const int row = quad * 32 + lane;  // TMEM lane = token row of the tile
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        constexpr int HM = MP / 2;
        const uint64_t pol_keep = policy_evict_last();
        uint32_t sidx = 0, ause = 0, iq = 0;  // ause: uses of the A buffers (pass-1 tiles)
        uint32_t own = 0;  // ping-pong: this group's uses of its A buffer
        uint32_t naw = 0;  // one A / W' buffer: pass-2 to pass-1 switches waited for
        bool after_p2 = false;
        bool ok = true;
        auto arrive_w = [&](uint64_t *bar) {  // one arrival per warp
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        while (ok) {
            if (!wait(iq_full + iq % kIQ, (iq / kIQ) & 1u)) break;
            const Item it = read_item(iq);
            sm_sync();
            if (tid == 0) mbar_arrive(iq_empty + iq % kIQ);
            ++iq;
            if (it.kind == kEnd) break;
            if (it.kind == kFlush) continue;
            int a1, b1;
            const int nt = item_tiles(it, p, a1, b1);
            for (int idx = 0; idx < nt && ok; ++idx) {
                const TileRef tr = tile_at(it, a1, b1, idx, p);
                if (LY::kAW && tr.kind == 1) after_p2 = true;
                if (tr.stored) continue;  // pass 2 of a split slice has no softmax
                if constexpr (LY::kPP) {
                    const int sb = (int)(sidx & 1u);
                    const uint32_t sph = (sidx >> 1) & 1u;
                    ++sidx;
                    const bool store = tr.kind == 0 && !tr.full && p.store_a;  // pass 2 reads A back
                    if (sb != g) {
                        // the other group's tile.  A chunk is published once every A row of it
                        // is stored: at its last tile this group's own stores are flushed too
                        if (store && tr.last && lane == 0) {
                            bulk_wait_group0();
                            fence_proxy_async_global();
                            red_release_cta_add(s_ast, 1u);
                        }
                        continue;
                    }
                    if (!wait(s_full + sb, sph)) { ok = false; break; }
                    tc_fence_after();
                    float v[MP], mg, zg;  // the whole row: the "half" of a 2 MP-wide row is MP columns
                    const uint32_t ts = trow + (sb ? LY::colS1 : LY::colS0);
                    if (p.m == MP) softmax_half<2 * MP, false>(ts, 0, p.m, p.c, v, mg, zg);
                    else softmax_half<2 * MP, true>(ts, 0, p.m, p.c, v, mg, zg);
                    tc_fence_before();
                    grp_sync(g);  // the group's four warps have read the S buffer
                    const bool valid = tr.tile * kT + row < p.n;
                    const uint64_t sc2 = f32x2(valid ? 1.f / zg : 0.f, valid ? 1.f / zg : 0.f);
                    uint32_t pk[MP / 2];
#pragma unroll
                    for (int j = 0; j < MP / 2; ++j) {
                        float x0, x1;
                        f32x2_split(mul_f32x2(f32x2(v[2 * j], v[2 * j + 1]), sc2), x0, x1);
                        pk[j] = pack_bf16x2(x0, x1);
                    }
                    if (tr.kind == 1) {  // pass 2: A over its S buffer, the H MMA's A operand in TMEM
                        tmem_st32(ts, pk);
                        tmem_st_wait();
                        tc_fence_before();
                        grp_sync(g);
                        if (quad == 0 && lane == 0) mbar_arrive(p_full + sb);
                        continue;
                    }
                    if (quad == 0 && lane == 0) mbar_arrive(s_empty + sb);
                    if (lane == 0) bulk_wait_group_read0();  // this warp's last A store has read buffer g
                    if (!wait(a_empty + g, (own & 1u) ^ 1u)) { ok = false; break; }
                    uint8_t *sAb = sA + g * LY::kAB;
#pragma unroll
                    for (int c8 = 0; c8 < MP / 8; ++c8)
                        *reinterpret_cast<uint4 *>(sAb + sw_off(row, c8, kT)) =
                            make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
                    fence_proxy_async_smem();
                    arrive_w(a_full + g);
                    ++own;
                    if (store && lane == 0) {
                        if (tr.tile * kT + quad * 32 < p.n) {
                            tma_store_3d(&ta_st, sAb + quad * 32 * 128, 0, tr.tile * kT + quad * 32, tr.slice, pol_keep);
                            bulk_commit_group();
                        }
                        if (tr.last) {
                            bulk_wait_group0();
                            fence_proxy_async_global();
                            red_release_cta_add(s_ast, 1u);
                        }
                    }
                    continue;
                }
                const int sb = (int)(sidx & 1u);
                if (!wait(s_full + sb, (sidx >> 1) & 1u)) { ok = false; break; }
                tc_fence_after();
                float v[HM], mg, zg;
                const uint32_t ts = trow + (sb ? LY::colS1 : LY::colS0) + g * HM;
                if (p.m == MP) softmax_half<MP, false>(ts, g * HM, p.m, p.c, v, mg, zg);
                else softmax_half<MP, true>(ts, g * HM, p.m, p.c, v, mg, zg);
                tc_fence_before();
                // this warp's last A store has read its rows before anyone rewrites them
                if (lane == 0) bulk_wait_group_read0();
                float2 *xc = sXch + (size_t)(sb * 2) * kT;
                xc[g * kT + row] = make_float2(mg, zg);
                sm_sync();  // both halves have read the S buffer
                // pass 1 frees the S buffer now; pass 2 writes its A over it, and the MMA that
                // consumes that A frees it
                if (tr.kind == 0 && tid == 0) mbar_arrive(s_empty + sb);
                const float2 o = xc[(g ^ 1) * kT + row];
                ++sidx;
                const float mrow = fmaxf(mg, o.x);
                const float own = ex2_approx((mg - mrow) * p.c), other = ex2_approx((o.x - mrow) * p.c);
                const bool valid = tr.tile * kT + row < p.n;
                const float scale = valid ? own / (zg * own + o.y * other) : 0.f;
                uint32_t pk[HM / 2];
                const uint64_t sc2 = f32x2(scale, scale);
#pragma unroll
                for (int j = 0; j < HM / 2; ++j) {
                    float x0, x1;
                    f32x2_split(mul_f32x2(f32x2(v[2 * j], v[2 * j + 1]), sc2), x0, x1);
                    pk[j] = pack_bf16x2(x0, x1);
                }
                if (tr.kind == 1) {
                    // pass 2: A (bf16 pairs) into the first MP/2 columns of the S buffer, the
                    // A operand of H = A W' straight from tensor memory
                    if (HM / 2 == 32) tmem_st32(ts - g * HM + g * (HM / 2), pk);
                    else tmem_st16(ts - g * HM + g * (HM / 2), pk);
                    tmem_st_wait();
                    tc_fence_before();
                    sm_sync();
                    if (tid == 0) mbar_arrive(p_full + sb);
                    continue;
                }
                const int ab = (int)(ause % NA);
                if (!wait(a_empty + ab, ((ause / NA) & 1u) ^ 1u)) { ok = false; break; }
                if (LY::kAW && after_p2) {  // the buffer held W': its pass-2 MMAs have completed
                    if (!wait(aw_a, naw & 1u)) { ok = false; break; }
                    ++naw;
                    after_p2 = false;
                }
                uint8_t *sAb = sA + ab * LY::kAB;
#pragma unroll
                for (int c8 = 0; c8 < HM / 8; ++c8)
                    *reinterpret_cast<uint4 *>(sAb + sw_off(row, g * (HM / 8) + c8, kT)) =
                        make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
                fence_proxy_async_smem();
                arrive_w(a_full + ab);
                ++ause;
                const bool store = tr.kind == 0 && !tr.full && p.store_a;  // pass 2 reads A back
                if (store) {
                    // MP = 128: each group stores its own 64-column block of its quadrant's 32
                    // rows; MP = 64: the block holds both halves, so the two warps of a quadrant
                    // meet first and group 0 stores it.  Rows past the end are not written.
                    if (MP == 64) asm volatile("bar.sync %0, 64;" ::"r"(5 + quad) : "memory");
                    if ((MP == 128 || g == 0) && lane == 0) {
                        if (tr.tile * kT + quad * 32 < p.n) {
                            const int b = MP == 128 ? g : 0;
                            tma_store_3d(&ta_st, sAb + b * kT * 128 + quad * 32 * 128, 64 * b, tr.tile * kT + quad * 32,
                                         tr.slice, pol_keep);
                            bulk_commit_group();
                        }
                        if (tr.last) {
                            // end of a chunk: its A rows are in global memory before the chunk is
                            // published (the epilogue waits for every storing warp)
                            bulk_wait_group0();
                            fence_proxy_async_global();
                            red_release_cta_add(s_ast, 1u);
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group0();  // no A store of this warp is still reading shared memory
    } else {
        // =========================================================== epilogue (warps 8-11)
        // H tiles out of TMEM to global; at the end of a pass-1 phase, the chunk partial and
        // its reduction (or, for whole slices, W' straight into shared memory).
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // TMEM lane: token row (H) / anchor row (W)
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t iq = 0, p2 = 0, wuse = 0, chunks = 0, lseq = 0, ew = 0;
        bool lpend = false;
        uint32_t accuse[2] = {0u, 0u};
        bool ok = true;
        auto arrive4 = [&](uint64_t *bar) {  // one arrival per warp
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        // bounded wait until the storing softmax warps (4, or 8 when MP = 128 or in ping-pong) have stored the
        // A rows of the chunks so far (a monotonic counter: no phase to alias)
        auto wait_ast = [&](uint32_t target) -> bool {
            if (ld_acquire_cta(s_ast) >= target) return true;
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_cta(s_ast) < target) {
                if (*s_abort) return false;
                if (globaltimer_ns() - t0 > kWaitNs) {
                    *s_abort = 1;
                    atomicOr(&g_umma_error, 1u);
                    return false;
                }
                __nanosleep(64);
            }
            return true;
        };
        const uint64_t pol_stream = policy_evict_first();
        int held = -1;  // ring slot whose H store may still be reading it (released one tile later)
        auto epilogue = [&](const TileRef &tr, int aslot) -> bool {
            if (tr.kind == 1) {
                // H tile -> bf16 -> a staging buffer -> TMA stores of 32 rows per warp
                const int hb = (int)(p2 & 1u);
                if (!wait(acc_full + hb, accuse[hb] & 1u)) return false;
                tc_fence_after();
                const uint32_t hcol = hb ? LY::colB1 : LY::colB0;
                const int r0 = tr.tile * kT + quarter * 32;
                if (LY::kStageH && !tr.stored) {
                    // the warp's own 4 KB buffer, one 64-column block of its 32 rows at a time:
                    // the block is read from TMEM and packed to bf16 before the wait for the
                    // buffer's last store
                    uint8_t *hs = sH + quarter * (32 * 128);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b) {
                        uint4 pk[8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float v[32];
                            tmem_ld32(trow + hcol + b * 64 + h * 32, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 4; ++c) pk[4 * h + c] = pack8_scaled(v + 8 * c, 1.f);
                        }
                        if (b == D / 64 - 1) {  // the accumulator is read: the next H MMA may start
                            tc_fence_before();
                            arrive4(acc_empty + hb);
                            ++accuse[hb];
                            ++p2;
                        }
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(hs + sw_off(lane, c, 32)) = pk[c];
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && r0 < p.n) {
                            tma_store_3d(&th_st, hs, 64 * b, r0, tr.slice, pol_stream);
                            bulk_commit_group();
                        }
                    }
                    return true;
                }
                // otherwise the ring slot that held this tile's A or Q, released after the stores
                // have read it
                uint8_t *stage = sRing + aslot * LY::kSlotB;
                // a deep ring lets the staging slot go back one tile later, so that this tile's
                // store reads it while the next tile is drained; the last tile of an item
                // releases both (the tile past the end, r0 >= n, is always an item's last)
                const bool defer = LY::kNSlot >= 6 && !tr.last;
                if constexpr (D == 64) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float v[32];
                        tmem_ld32(trow + hcol + q * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4 *>(stage + sw_off(row, q * 4 + c, kT)) = pack8_scaled(v + 8 * c, 1.f);
                    }
                    tc_fence_before();
                    arrive4(acc_empty + hb);
                    ++accuse[hb];
                    ++p2;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && r0 < p.n) tma_store_3d(&th_st, stage + quarter * 32 * 128, 0, r0, tr.slice, pol_stream);
                } else {
                    // per 64-column block: two TMEM loads behind one wait, then the block's
                    // store goes out while the next block is drained
#pragma unroll
                    for (int b = 0; b < D / 64; ++b) {
                        float v[64];
                        tmem_ld32(trow + hcol + b * 64, v);
                        tmem_ld32(trow + hcol + b * 64 + 32, v + 32);
                        tmem_ld_wait();
                        if (b == D / 64 - 1) {  // the accumulator is read: the next H MMA may start
                            tc_fence_before();
                            arrive4(acc_empty + hb);
                            ++accuse[hb];
                            ++p2;
                        }
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(stage + sw_off(row, b * 8 + c, kT)) = pack8_scaled(v + 8 * c, 1.f);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && r0 < p.n)
                            tma_store_3d(&th_st, stage + b * kT * 128 + quarter * 32 * 128, 64 * b, r0, tr.slice, pol_stream);
                    }
                }
                if (lane == 0) {
                    if (r0 < p.n) bulk_commit_group();
                    if (defer) bulk_wait_group_read1();
                    else bulk_wait_group_read0();  // also covers the held slot's store
                }
                const int tok = tr.tile * kT + row;
                if (tr.stored && tok < p.n) {
                    // the H MMA has read this A row: nothing reads it again, so its L2 lines
                    // are dropped instead of being written back to memory
                    const uint8_t *arow = reinterpret_cast<const uint8_t *>(p.abuf + ((size_t)tr.slice * p.n + tok) * MP);
#pragma unroll
                    for (int l = 0; l < MP * 2 / 128; ++l) discard_l2_line(arow + 128 * l);
                }
                ep_sync();
                if (row == 0) {
                    if (held >= 0) mbar_arrive(slot_empty + held);  // the last tile's store has read it
                    if (!defer) mbar_arrive(slot_empty + aslot);
                }
                held = defer ? aslot : -1;
                return true;
            }
            if (!tr.last) return true;
            // end of a pass-1 phase: W (anchor row `row`, D columns) and Delta in TMEM
            const int wbuf = (int)(ew & 1u);
            if constexpr (LY::kWSep) {
                if (!wait(wacc_full + wbuf, (ew >> 1) & 1u)) return false;
            } else {
                if (!wait(acc_full + 0, accuse[0] & 1u)) return false;
                if (!wait(acc_full + 1, accuse[1] & 1u)) return false;
            }
            const uint32_t wcol = wbuf ? LY::colW1 : LY::colW0;
            auto release_w = [&]() {  // the chunk accumulators are read
                if constexpr (LY::kWSep) {
                    arrive4(wacc_empty + wbuf);
                } else {
                    arrive4(acc_empty + 0);
                    arrive4(acc_empty + 1);
                    ++accuse[0];
                    ++accuse[1];
                }
                ++ew;
            };
            tc_fence_after();
            float v[32];
            tmem_ld32(trow + wcol + D, v);
            tmem_ld_wait();
            const float dj = v[0];
            if (!tr.full) {
                // this chunk's W row -> workspace (before TMEM is released to the next MMAs)
                if (row < MP) {
                    // partial layout [D/4][MP] float4: a warp's 32 anchors write 512 contiguous bytes
                    float4 *dst = reinterpret_cast<float4 *>(p.part + ((size_t)tr.slice * p.C1 + tr.chunk) * MP * D) + row;
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        tmem_ld32(trow + wcol + q * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[(q * 8 + i) * MP] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                    p.pdelta[((size_t)tr.slice * p.C1 + tr.chunk) * MP + row] = dj;
                } else {
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) tmem_ld32(trow + wcol + q * 32, v);  // keep the warp converged
                    tmem_ld_wait();
                }
                tc_fence_before();
                release_w();
                ++chunks;
                bool published = false;
                // Fixed binary tree over the slice's chunks: node (l, i) covers chunks
                // [i 2^(l+1), (i+1) 2^(l+1)).  The second of its two children to arrive forms
                // left + right into the left child's slot and climbs on; the first stops.  The
                // sums - and so W - do not depend on which CTA arrived first.
                for (int l = 0; (1 << l) < p.C1; ++l) {
                    const int left = (tr.chunk >> (l + 1)) << (l + 1), right = left + (1 << l);
                    if (right >= p.C1) continue;  // no right subtree at this level
                    // the group's partial writes are ordered before thread 0's release by the
                    // barrier; its acquire orders the sibling's partial before the group's reads
                    ep_sync();
                    if (row == 0) {
                        // this chunk's A rows must be in memory before the chunk is published;
                        // if that wait gives up (abort), stop here as if first to arrive
                        const bool go = published || !p.store_a || wait_ast((MP == 128 || LY::kPP ? 8u : 4u) * chunks);
                        published = true;
                        *s_last = go ? (int)atom_add_acq_rel_gpu(p.tree + (size_t)tr.slice * p.C1 + (right - 1), 1u) : 0;
                    }
                    ep_sync();
                    if (*s_last == 0) return true;  // first to arrive: the sibling's CTA goes on
                    const bool root = (2 << l) >= p.C1;
                    if (row < MP) {
                        const size_t dl_ = ((size_t)tr.slice * p.C1 + left) * MP + row;
                        const size_t dr_ = ((size_t)tr.slice * p.C1 + right) * MP + row;
                        const float dsum = __ldcg(p.pdelta + dl_) + __ldcg(p.pdelta + dr_);
                        const float4 *sl = reinterpret_cast<const float4 *>(p.part + ((size_t)tr.slice * p.C1 + left) * MP * D) + row;
                        const float4 *sr = reinterpret_cast<const float4 *>(p.part + ((size_t)tr.slice * p.C1 + right) * MP * D) + row;
                        float4 *dl = reinterpret_cast<float4 *>(p.part + ((size_t)tr.slice * p.C1 + left) * MP * D) + row;
                        const float rinv = dsum != 0.f ? 1.f / dsum : 0.f;
                        uint8_t *img = reinterpret_cast<uint8_t *>(p.wimg + (size_t)tr.slice * (D * MP));
                        // 4 groups of D/16 float4 from each side (8-column chunks stay whole)
                        constexpr int QV = D / 16;
#pragma unroll 1
                        for (int g = 0; g < 4; ++g) {
                            float4 xl[QV], xr[QV];
#pragma unroll
                            for (int i = 0; i < QV; ++i) {
                                xl[i] = __ldcg(sl + (g * QV + i) * MP);
                                xr[i] = __ldcg(sr + (g * QV + i) * MP);
                            }
#pragma unroll
                            for (int i = 0; i < QV; ++i)
                                xl[i] = make_float4(xl[i].x + xr[i].x, xl[i].y + xr[i].y, xl[i].z + xr[i].z, xl[i].w + xr[i].w);
                            if (!root) {
#pragma unroll
                                for (int i = 0; i < QV; ++i) dl[(g * QV + i) * MP] = xl[i];
                            } else {  // every chunk is in: W'_jk = W_jk / Delta_j, bf16 image
#pragma unroll
                                for (int i = 0; i < QV; i += 2) {
                                    const float w8[8] = {xl[i].x, xl[i].y, xl[i].z, xl[i].w,
                                                         xl[i + 1].x, xl[i + 1].y, xl[i + 1].z, xl[i + 1].w};
                                    *reinterpret_cast<uint4 *>(img + wimg_chunk_off<MP>(row, (g * QV + i) / 2)) =
                                        pack8_scaled(w8, rinv);
                                }
                            }
                        }
                        if (!root) p.pdelta[dl_] = dsum;
                    }
                    if (root) {
                        // the image is read by bulk copies: order it for the async proxy; the
                        // flag's release (after the barrier) publishes every thread's writes
                        fence_proxy_async_global();
                        ep_sync();
                        if (row == 0 && tr.slice != p.hold_slice) st_release_gpu(p.flags + 32 * tr.slice, 1u);
                        return true;
                    }
                }
                return true;
            }
            // whole slice on chip: W' = Delta^{-1} W straight into the shared operand image
            const int wb = (int)(wuse % NW);
            uint8_t *sWb = sW + wb * LY::kWB;
            if (!wait(w_empty + wb, ((wuse / NW) & 1u) ^ 1u)) return false;
            const float rinv = dj != 0.f ? 1.f / dj : 0.f;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                tmem_ld32(trow + wcol + q * 32, v);
                tmem_ld_wait();
                if (row < MP) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(sWb + wimg_chunk_off<MP>(row, q * 4 + c)) = pack8_scaled(v + 8 * c, rinv);
                }
            }
            tc_fence_before();
            release_w();
            fence_proxy_async_smem();
            ep_sync();
            if (row == 0) mbar_arrive(w_full + wb);
            return true;
        };

        while (ok) {
            if (!wait(iq_full + iq % kIQ, (iq / kIQ) & 1u)) break;
            const Item it = read_item(iq);
            ep_sync();
            if (row == 0) mbar_arrive(iq_empty + iq % kIQ);
            ++iq;
            if (it.kind == kEnd) break;
            // the ring positions, replayed from the item stream exactly as the producer fills
            // them: one slot per tile (Q, or the stored A), then the previous pass-1 tile's V
            if (it.kind == kFlush) {
                if (lpend) ++lseq;
                lpend = false;
                continue;
            }
            int a1, b1;
            const int nt = item_tiles(it, p, a1, b1);
            for (int idx = 0; idx < nt && ok; ++idx) {
                const TileRef tr = tile_at(it, a1, b1, idx, p);
                const int aslot = (int)(lseq % NS);
                ++lseq;
                if (LY::kVLag) {
                    if (lpend) ++lseq;
                    lpend = tr.kind == 0;
                } else if (tr.kind == 0) {
                    ++lseq;  // this tile's V
                }
                if (!epilogue(tr, aslot)) { ok = false; break; }
                if (tr.kind == 1 && tr.first) ++wuse;  // W' uses started so far
            }
        }
        if (lane == 0) bulk_wait_group0();  // this warp's H stores have left shared memory
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMmaS) {
        tc_fence_after();
        tmem_dealloc(tmem, LY::kTmemCols);
    }
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
cudaError_t launch_t(const Problem &pr, const UmmaPlan &pl, const UmmaOptions &opt, void *ws, cudaStream_t stream) {
    static_assert(Layout<D, MP>::kSmem <= 227 * 1024, "shared memory");
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

    CUtensorMap tq, tv, tu, ta_st, ta_ld;
    const long long S = pr.slices();
    if (!make_map(&tq, pr.Q, D, pr.n, S, kT) || !make_map(&tv, pr.V, D, pr.n, S, kT) ||
        !make_map(&tu, pr.U, D, pr.m, pr.heads, MP))
        return cudaErrorInvalidValue;

    UParams p;
    p.slices = (int)S;
    p.heads = pr.heads;
    p.B = pr.B;
    p.n = pr.n;
    p.m = pr.m;
    p.c = pr.scale * 1.4426950408889634f;
    p.NT = pl.NT;
    p.C1 = pl.C1;
    p.C2 = pl.C2;
    p.S2f = pl.S2f;
    p.C2f = pl.C2f;
    const int grid = (int)std::min<long long>((long long)sms * per_sm, pl.total_items);
    uint8_t *w = static_cast<uint8_t *>(ws);
    // header (zeroed each call): next | head | flags[S] and P2 claim counters[S], one 128-byte
    // line each | tree arrival counters [S][C1]
    p.next = reinterpret_cast<unsigned *>(w);
    p.head = reinterpret_cast<unsigned *>(w + 128);
    p.flags = reinterpret_cast<unsigned *>(w + 256);
    p.p2c = p.flags + 32 * S;
    p.tree = p.p2c + 32 * S;
    // P1 runs at most K slices ahead of P2, so that the A tiles of the slices in flight
    // (written in pass 1, read in pass 2) fit in a share of L2
    p.store_a = pl.store_a ? 1 : 0;
    const double kept_slice = (double)pr.n * (pl.store_a ? MP : D) * 2;  // A copy, or Q for its re-read
    p.K = (int)std::max<double>(2.0, std::min<double>((double)S, 2.0 * (double)l2_bytes() / kept_slice));
    p.p1first = p.K >= S ? 1 : 0;
    p.hold_slice = opt.hold_slice;
    p.wait_ns = opt.wait_ns;
    uint8_t *after = w + pl.header_bytes;
    p.pdelta = reinterpret_cast<float *>(after);
    p.part = p.pdelta + (size_t)S * pl.C1 * MP;
    p.wimg = reinterpret_cast<uint16_t *>(p.part + (size_t)S * pl.C1 * D * MP);
    p.abuf = reinterpret_cast<uint16_t *>(w + pl.abuf_offset);
    if (pl.C1 == 1) p.part = p.pdelta = nullptr, p.wimg = nullptr;
    if (!pl.store_a) p.abuf = nullptr;
    // the stored A: row-major [S][n][MP]; pass 1 stores 32-row slabs (one per softmax warp),
    // pass 2 loads 128-row tiles.  Whole-slice plans have no stored A: the maps then point
    // at Q, which is never touched through them.
    const void *abase = p.abuf ? static_cast<const void *>(p.abuf) : pr.Q;
    if (!make_map(&ta_st, abase, MP, pr.n, p.abuf ? S : 1, 32) || !make_map(&ta_ld, abase, MP, pr.n, p.abuf ? S : 1, kT))
        return cudaErrorInvalidValue;
    CUtensorMap th_st;  // H rows, 32-row boxes (one per epilogue warp)
    if (!make_map(&th_st, pr.H, D, pr.n, S, 32)) return cudaErrorInvalidValue;

    if ((e = cudaMemsetAsync(ws, 0, pl.header_bytes, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, LY::kSmem, stream>>>(tq, tv, tu, ta_st, ta_ld, th_st, p, static_cast<uint16_t *>(pr.H));
    return cudaGetLastError();
}

}  // namespace

bool make_bf16_map(CUtensorMap *map, const void *base, int cols, int rows, long long outer, int box_rows) {
    return make_map(map, base, cols, rows, outer, box_rows);
}

// L2 size of the current device (126 MiB, GB300's, when no device can be queried: plans are
// also asked for on machines without one)
size_t l2_bytes() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return size_t(126) << 20;
    }
    return (size_t)n;
}

UmmaPlan umma_plan(const Problem &p, bool force_recompute) {
    UmmaPlan pl;
    const int MP = p.m <= 64 ? 64 : 128;
    pl.MP = MP;
    pl.NT = (p.n + kT - 1) / kT;
    const long long S = p.slices();
    // Chunk sizes: long chunks mean fewer partials to reduce, fewer anchor reloads and fewer
    // item switches, but every SM needs work: halve a pass's chunk while the pass has fewer
    // than one and a half items per SM.  The SM count assumed here is a constant, not the
    // device's, so that the chunks - and so the summation order and the result bits - depend
    // on the shape alone.
    const long long want = 3LL * kPlanSMs / 2;
    int t1 = kUmmaP1Tiles, t2 = kUmmaP2Tiles;
    // (pass 1's chunks set the summation order of W: they follow the plan's slice count)
    while (t1 > kUmmaMinTiles && p.plan_S() * ((pl.NT + t1 - 1) / t1) < want) t1 /= 2;
    while (t2 > kUmmaMinTiles && S * ((pl.NT + t2 - 1) / t2) < want) t2 /= 2;
    pl.C1 = (pl.NT + t1 - 1) / t1;
    // Pass 2 reuses pass 1's A only when every slice's copy fits in half of a GB300's L2
    // together (kStoreABytes); otherwise the copy would make a round trip through memory, and
    // recomputing A from Q costs less.  The chunking does not depend on which of the two runs
    // (nor on a forced recompute, a test option), and the stored and the recomputed A are the
    // same bf16 values: every plan of a shape gives the same bits.
    const bool store_a = !force_recompute && 2.0 * (double)S * p.n * MP <= (double)kStoreABytes;
    if (pl.NT <= kUmmaFullTiles || pl.C1 == 1) {
        pl.C1 = 1;
        pl.C2 = 0;
        pl.total_items = (int)S;
        pl.header_bytes = 256;
        pl.workspace_bytes = 256;
        return pl;
    }
    pl.C2 = (pl.NT + t2 - 1) / t2;
    // the last slices' pass 2 in chunks kUmmaFineSplit times finer: about a quarter of a wave
    // (one pass-2 item per SM) of slices, which the SMs freed first share out at the end
    // (long_16k: 207.0 -> 203.5 us; half a wave 204.8, a whole wave 207.0, four times finer
    // 208.4)
    pl.C2f = std::min(pl.NT, pl.C2 * kUmmaFineSplit);
    const long long fine = std::min<long long>(S, ((long long)kPlanSMs * t2 / 4 + pl.NT - 1) / pl.NT);
    pl.S2f = (int)(S - (pl.C2f > pl.C2 ? fine : 0));
    pl.total_items = (int)(S * pl.C1 + (long long)pl.S2f * pl.C2 + (S - pl.S2f) * (long long)pl.C2f);
    pl.header_bytes = (256 + 2 * 128 * (size_t)S + 4 * (size_t)S * pl.C1 + 1023) / 1024 * 1024;
    const size_t reduce_bytes = 4 * (size_t)S * pl.C1 * MP + 4 * (size_t)S * pl.C1 * p.d * MP + 2 * (size_t)S * p.d * MP;
    pl.abuf_offset = (pl.header_bytes + reduce_bytes + 1023) / 1024 * 1024;
    pl.store_a = store_a;
    pl.workspace_bytes = pl.abuf_offset + (pl.store_a ? 2 * (size_t)S * p.n * MP : 0);
    return pl;
}

bool umma_supported(const Problem &p) {
    // scale > 0: the softmax takes the row maximum of the raw scores
    return !p.f32 && (p.d == 64 || p.d == 128) && p.m >= 32 && p.m <= 128 && p.scale > 0.f &&
           p.slices() * ((p.n + kT - 1) / kT) * 3 < 0x7fffffffLL;
}

cudaError_t launch_umma(const Problem &p, const UmmaPlan &pl, const UmmaOptions &opt, void *workspace,
                        cudaStream_t stream) {
    if (p.d == 64 && pl.MP == 64) return launch_t<64, 64>(p, pl, opt, workspace, stream);
    if (p.d == 64 && pl.MP == 128) return launch_t<64, 128>(p, pl, opt, workspace, stream);
    if (p.d == 128 && pl.MP == 64) return launch_t<128, 64>(p, pl, opt, workspace, stream);
    if (p.d == 128 && pl.MP == 128) return launch_t<128, 128>(p, pl, opt, workspace, stream);
    return cudaErrorInvalidValue;
}

cudaError_t umma_read_and_clear_error(unsigned *out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_umma_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_umma_error, &zero, sizeof(unsigned));
}

}  // namespace anchor

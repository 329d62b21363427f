// Shared device helpers and the internal launch interface of the anchor-attention kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "anchor_attn.h"

namespace anchor {

// One forward problem as the C ABI received it (device pointers, validated).
struct Problem {
    const void *Q;
    const void *U;
    const void *V;
    void *H;
    int B, heads, n, m, d;
    float scale;
    bool f32;  // element type of Q, U, V, H: float (true) or bf16 (false)
    // the slice count the persistent tensor-core plan cuts a slice's pass 1 by (its chunks set
    // the summation order of W): 0 = this problem's own.  A part of a larger problem run on its
    // own (the host entry's chunks) passes the whole problem's, so that its bits match the
    // whole problem's.
    long long plan_slices = 0;
    // the slice-streaming kernel's CTAs per slice; 0 = what this problem's shape gives.  The
    // host entry's chunks pass the whole problem's.
    int plan_cl_c = 0;
    long long slices() const { return (long long)B * heads; }
    long long plan_S() const { return plan_slices > 0 ? plan_slices : slices(); }
};
// the forward of a problem (the C ABI's checks, plan and launch; used by the host entry)
anchor_attn_status_t forward_problem(const Problem &p, void *stream);
// the CTAs per slice the forward of `p` runs the slice-streaming kernel with; 0 when it takes
// another kernel
int forward_stream_cluster(const Problem &p);

// Argument checks of the C ABI (see include/anchor_attn.h); no device access.
anchor_attn_status_t check_shape(int B, int heads, int n, int m, int d);
anchor_attn_status_t check_problem(const Problem &p);

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Butterfly sum: every lane ends with the same value, in an order fixed by the lane
// pattern, so the result is the same from run to run.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// --- SIMT (CUDA-core) variants -------------------------------------------------------
constexpr int kSimtChunk = 512;                  // tokens per pass-1 chunk of the chunked kernel
constexpr size_t kSimtMaxSmem = 220 * 1024;      // dynamic shared memory a CUDA-core CTA may use
constexpr size_t kSimtThirdSmem = 72 * 1024;     // ... when three such CTAs are to share an SM
// workspace of the chunked kernel: a zeroed header (ticket, per-slice arrival counters and
// ready flags), the chunk partials [slices][chunks][m d + m] fp32 and W' [slices][m d] fp32
struct SimtLayout {
    size_t header_bytes = 0, part_offset = 0, wprime_offset = 0, total_bytes = 0;
};
bool simt_full_fits(const Problem &p);     // the whole slice fits one CTA's shared memory
bool simt_chunk_fits(const Problem &p);    // the chunked kernel's anchors and tiles fit
SimtLayout simt_chunk_layout(const Problem &p);
cudaError_t launch_simt_full(const Problem &p, cudaStream_t stream);
cudaError_t launch_simt_chunk(const Problem &p, void *workspace, cudaStream_t stream);
cudaError_t simt_read_and_clear_error(unsigned *out);

// --- backward (CUDA-core) -------------------------------------------------------------
struct BwdProblem {
    const void *Q, *U, *V, *dH;
    void *dQ, *dU, *dV;
    int B, heads, n, m, d;
    float scale;
    bool f32;
    long long slices() const { return (long long)B * heads; }
};
// workspace: a zeroed header (ticket, arrival counters, ready flags), the chunk partials
// [slices][chunks][m + 2 m d], the published W' | dW | dDelta per slice, and the chunks' dU
// shares [slices][chunks][m d] (all fp32)
struct BwdLayout {
    size_t header_bytes = 0, part_offset = 0, pub_offset = 0, dupart_offset = 0, total_bytes = 0;
};
bool bwd_fits(const BwdProblem &p);
BwdLayout bwd_layout(const BwdProblem &p);
cudaError_t launch_bwd(const BwdProblem &p, void *workspace, cudaStream_t stream);
cudaError_t bwd_read_and_clear_error(unsigned *out);
// dU[h] = sum over batch entries b, then chunks c, of dupart[b heads + h][c] ([m d] fp32 blocks)
cudaError_t launch_bwd_du_sum(const float *dupart, void *dU, int B, int heads, int chunks, int md, bool f32,
                              cudaStream_t stream);
// the backward on the tensor cores (bf16, d = 64, m <= 64): workspace = the slices' dU blocks
bool bwd_tc_supported(const BwdProblem &p);
size_t bwd_tc_workspace(const BwdProblem &p);
cudaError_t launch_bwd_tc(const BwdProblem &p, void *workspace, cudaStream_t stream);
cudaError_t bwd_tc_read_and_clear_error(unsigned *out);
// the backward on the tensor cores for d = 64 or 128, m <= 128 (bf16): pass 1, a per-slice
// reduce, pass 2 and the dU sum over runs of each slice's tiles; workspace = the items' pass-1
// blocks, the slices' W' and dW images, dDelta and the items' dU blocks.  Preferred for d = 128
// and for d = 64 with m > 64; d = 64 with m <= 64 takes bwd_tc.
bool bwd_wide_supported(const BwdProblem &p);
bool bwd_wide_preferred(const BwdProblem &p);
size_t bwd_wide_workspace(const BwdProblem &p);
cudaError_t launch_bwd_wide(const BwdProblem &p, void *workspace, cudaStream_t stream);
cudaError_t bwd_wide_read_and_clear_error(unsigned *out);

// --- masked (causal) variant (CUDA-core) ------------------------------------------------
// workspace: a zeroed header, the chunks' totals [slices][chunks][m + m d] and their
// exclusive prefixes [slices][chunks][m d + m rounded up to 4] (fp32)
struct CausalLayout {
    size_t header_bytes = 0, part_offset = 0, pre_offset = 0, total_bytes = 0;
};
bool causal_fits(const Problem &p);
CausalLayout causal_layout(const Problem &p);
cudaError_t launch_causal(const Problem &p, void *workspace, cudaStream_t stream);
cudaError_t causal_read_and_clear_error(unsigned *out);
// the masked variant on the tensor cores (bf16, d = 64, m <= 64; no workspace)
bool causal_tc_supported(const Problem &p);
cudaError_t launch_causal_tc(const Problem &p, cudaStream_t stream);
cudaError_t causal_tc_read_and_clear_error(unsigned *out);
// the masked variant on the tensor cores for up to 128 anchors (d = 128, or d = 64 with m > 64)
bool causal_wide_supported(const Problem &p);
cudaError_t launch_causal_wide(const Problem &p, cudaStream_t stream);
cudaError_t causal_wide_read_and_clear_error(unsigned *out);

// --- approximation-error diagnostic ------------------------------------------------------
struct FullProblem {
    const void *Q, *K, *V;  // K: [heads][n][d], one key matrix per head shared by the batch
    void *H;
    int B, heads, n, d;
    float scale;
    bool f32;
    long long slices() const { return (long long)B * heads; }
};
cudaError_t launch_full_attention(const FullProblem &p, cudaStream_t stream);
cudaError_t launch_rel_error(const void *Href, const void *H, float *err, long long slices, size_t per_slice, bool f32,
                             cudaStream_t stream);

// --- block front end (tensor core): Q and V projected from the token embeddings -------------
struct BlockProblem {
    const void *X;          // [B][n][dm] bf16 token embeddings
    const void *Wq, *Wv;    // [heads][d][dm] bf16 rows of the query / value projections
    const void *U;          // [heads][m][d] bf16 anchors
    void *H;                // [B][heads][n][d] bf16
    int B, heads, n, m, d, dm;
    float scale;
};
bool block_supported(const BlockProblem &p);
cudaError_t launch_block(const BlockProblem &p, cudaStream_t stream);
// the plain forward on short slices (bf16, d = 64, m <= 64, n <= 256) with the same kernel:
// one CTA per slice, two per SM, no workspace
bool short_supported(const Problem &p);
cudaError_t launch_short(const Problem &p, cudaStream_t stream);
cudaError_t block_read_and_clear_error(unsigned *out);

// 3-D bf16 tensor map [outer][rows][cols], box 64 columns x box_rows rows x 1, 128-byte swizzle
// Programmatic dependent launch.  A kernel launched with programmatic stream serialization
// may start while the kernel before it in the stream is still running.  It touches global
// memory only after grid_dependency_wait() (which returns once that kernel has completed and
// its writes are visible), and lets the next such launch start early with
// grid_dependents_launch().
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Launch with programmatic stream serialization: the kernel's setup may overlap the end of the
// previous kernel in the stream; the kernel itself waits (grid_dependency_wait) before it
// touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

bool make_bf16_map(CUtensorMap *map, const void *base, int cols, int rows, long long outer, int box_rows);

// --- slice-streaming tensor-core variant (d = 64, m <= 64): one CTA per slice ----------------
// workspace: the A tiles of pass 1, [slices][n][64] bf16
bool stream_supported(const Problem &p);
int stream_cluster(const Problem &p);  // CTAs per slice (a cluster when more than 1)
size_t stream_workspace(const Problem &p);
cudaError_t launch_stream(const Problem &p, void *workspace, cudaStream_t stream);
cudaError_t stream_read_and_clear_error(unsigned *out);

// --- split tensor-core variant (d = 64, m <= 64): the slices' tiles cut over kPlanSMs CTAs --------
// workspace: the A tiles [slices][n][64] bf16 first (so that launch_stream can run on it),
// then a zeroed header (per-slice counters and flags), the parts' (W, Delta) partials and the
// slices' W' images.  launch_split returns cudaErrorCooperativeLaunchTooLarge when the device
// cannot hold all kPlanSMs CTAs at once.
bool split_supported(const Problem &p);
size_t split_workspace(const Problem &p);
cudaError_t launch_split(const Problem &p, void *workspace, cudaStream_t stream);
cudaError_t split_read_and_clear_error(unsigned *out);

// --- tensor-core (tcgen05) variant ---------------------------------------------------
constexpr int kUmmaFullTiles = 4;    // slices of <= 4 tiles (512 tokens) run whole in one CTA
constexpr int kUmmaP1Tiles = 32;     // tiles per pass-1 chunk (halved while items are too few)
constexpr int kUmmaP2Tiles = 16;     // tiles per pass-2 chunk (halved while items are too few)
constexpr int kUmmaMinTiles = 4;     // smallest chunk either pass is cut into
constexpr int kUmmaFineSplit = 2;    // pass-2 chunks of the last slices: this many times finer
constexpr int kPlanSMs = 152;        // SM count the chunking assumes on every device
constexpr double kStoreABytes = 64.0 * 1024 * 1024;  // largest A copy (all slices) pass 2 reads back
struct UmmaPlan {
    int MP = 0;              // anchors padded to 64 or 128
    int NT = 0;              // 128-token tiles per slice
    int C1 = 0, C2 = 0;      // chunks per slice in pass 1 / pass 2 (C1 == 1: whole slice per CTA)
    int S2f = 0, C2f = 0;    // slices from schedule index S2f on take C2f pass-2 chunks
    int total_items = 0;
    size_t header_bytes = 0; // zeroed part of the workspace (ticket, counters, flags)
    size_t abuf_offset = 0;  // the A copy pass 2 reads: [slices][n][MP] bf16 (split slices only)
    bool store_a = false;    // pass 2 loads the A copy (else it recomputes A from Q)
    size_t workspace_bytes = 0;
};
// Run-time options of one tensor-core launch.
struct UmmaOptions {
    int hold_slice = -1;                      // failure-detection tests: never publish this slice's W'
    unsigned long long wait_ns = 2000000000ull;  // limit of a wait on other CTAs
};
bool umma_supported(const Problem &p);
UmmaPlan umma_plan(const Problem &p, bool force_recompute = false);
size_t l2_bytes();
cudaError_t launch_umma(const Problem &p, const UmmaPlan &plan, const UmmaOptions &opt, void *workspace,
                        cudaStream_t stream);
cudaError_t umma_read_and_clear_error(unsigned *out);

}  // namespace anchor

/*
 * anchor_attn.h - C ABI of the GB300 (sm_103a) anchor-attention forward.
 *
 * The operation (AnchorFormer, arXiv 2505.16463; pith.science verdict on 2505.16463,
 * "core_discovery", "key_machinery" and the referee summary of Eq. 11/12):
 *
 *   A[i][j] = softmax over j of ( scale * q_i . u_j )      n x m, rows sum to one
 *   Delta   = diag( sum_i A[i][j] )                        m x m, the anchor degrees
 *   H       = A Delta^{-1} A^T V                           n x d
 *
 * evaluated as A (Delta^{-1} (A^T V)), so no n x n matrix exists anywhere (the reordering
 * B^T V -> Delta^{-1}(B^T V) -> B(Delta^{-1} B^T V) of the referee summary, B == A).
 * Each (batch, head) pair - a "slice" - is independent (the construction is per head).
 * An anchor that no token reaches (Delta_j == 0 after underflow) contributes nothing.
 *
 * Layout (row-major, dense, no padding):
 *   Q, V, H : [B][heads][n][d]
 *   U       : [heads][m][d]    one set of m learnable anchor keys per head, shared by
 *                              every batch entry
 * Every pointer is a DEVICE pointer, 16-byte aligned.  The caller owns all buffers.
 * H must not overlap Q, U or V (the forward reads Q twice).
 *
 * Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as void*;
 * NULL = the legacy default stream).  No host synchronisation happens inside.
 * Workspace, where a variant needs one, is taken with cudaMallocAsync on `stream` and
 * released with cudaFreeAsync on the same stream before the call returns.
 * Results are bit-identical from run to run with the same library build: the way the tokens
 * of a slice are cut into chunks, and so the order of every sum, depends on the shape alone
 * (not on the device's SM or L2 size, nor on which CTA ran what).
 *
 * Shapes: B, heads, n >= 0 (a zero makes the call a no-op that returns OK and accepts NULL
 * pointers); m >= 1; d in {16, 32, 64, 128}; m * d <= 16384 (so m <= 256 for d <= 64 and
 * m <= 128 for d = 128); B * heads * n * d < 2^63.  scale must be finite.
 *
 * Errors are returned, never thrown or printed; a failed call launches nothing unless the
 * status is ANCHOR_ATTN_ERR_CUDA.
 */
#ifndef ANCHOR_ATTN_H
#define ANCHOR_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ANCHOR_ATTN_API __attribute__((visibility("default")))
#else
#define ANCHOR_ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ANCHOR_ATTN_OK = 0,
    ANCHOR_ATTN_ERR_INVALID_ARG = 1, /* NULL or misaligned pointer, negative size, m < 1,
                                        non-finite scale, size overflow                   */
    ANCHOR_ATTN_ERR_UNSUPPORTED = 2, /* d not in {16,32,64,128}, or m * d > 16384         */
    ANCHOR_ATTN_ERR_ALIAS = 3,       /* H overlaps Q, U or V                               */
    ANCHOR_ATTN_ERR_ALLOC = 4,       /* workspace allocation failed                        */
    ANCHOR_ATTN_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed               */
    ANCHOR_ATTN_ERR_SCRATCH_LIMIT = 6 /* the problem needs more scratch than the fixed
                                         array of anchor_attn_forward_static_scratch holds */
} anchor_attn_status_t;

/*
 * bf16 forward: Q, U, V, H are bf16 (uint16 bit patterns of bfloat16); scores, softmax,
 * Delta and every contraction accumulate in fp32; H is rounded to bf16 (nearest even).
 * On d in {64, 128} with 32 <= m <= 128 the three n x m x d contractions run on the
 * tensor cores (tcgen05, bf16 operands, fp32 accumulators in tensor memory); elsewhere on
 * CUDA-core fp32 FMA.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_forward(const void *Q, const void *U, const void *V, void *H,
                                         int B, int heads, int n, int m, int d, float scale,
                                         void *stream);

/*
 * fp32 forward: float in, float out, fp32 CUDA-core arithmetic throughout (expf, fixed-order
 * fp32 sums).  Same layout, shapes and errors as anchor_attn_forward.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_forward_f32(const float *Q, const float *U, const float *V,
                                             float *H, int B, int heads, int n, int m, int d,
                                             float scale, void *stream);

/*
 * Forward from host buffers: Q, U, V and H are host pointers (pinned memory, e.g. from
 * cudaHostAlloc, for the copies to run asynchronously; pageable memory works but the copies
 * then hold the calling thread), same layout, shapes, numbers and errors as
 * anchor_attn_forward.  The batch is cut into chunks of whole batch entries, or of head ranges
 * of single batch entries when that gives too few chunks; chunk by chunk Q and V are copied to
 * the device on an internal stream, the forward runs on `stream`, and H is copied back on a
 * second internal stream, over two device buffer sets, so that copies in, forward and copies
 * out of neighbouring chunks overlap.  The results are bit-identical to anchor_attn_forward's
 * (the same kernels, planned for the whole problem), except where the whole problem has more
 * than 152 slices at d = 64 with 32 <= m <= 64 and n > 512: there the device entry cuts the
 * tile list over the SMs and the chunks do not, so sums run in another order (the same values
 * within rounding).  Asynchronous: H is complete once `stream` has reached
 * this point (every internal copy is ordered before it); work already on `stream` is ordered
 * before the copies.  The device workspace (U and two chunks of Q, V, H) comes from
 * cudaMallocAsync on `stream` and goes back on it (ANCHOR_ATTN_ERR_ALLOC if it cannot be
 * had).  Calls on one device take a lock while they enqueue.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_forward_host(const void *Q, const void *U, const void *V, void *H,
                                                              int B, int heads, int n, int m, int d, float scale,
                                                              void *stream);
/* fp32 forward from host buffers (as anchor_attn_forward_f32, same pipeline). */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_forward_host_f32(const float *Q, const float *U, const float *V,
                                                                  float *H, int B, int heads, int n, int m, int d,
                                                                  float scale, void *stream);

/*
 * Backward of anchor_attn_forward, bf16 in and out, fp32 accumulation.  The
 * anchors are fitted by gradient descent (pith.science verdict on arXiv 2505.16463,
 * "core_discovery"; the arXiv abstract, where the anchors are weights of a trainable layer), so a layer
 * built on the forward needs the gradients of a loss L with respect to Q, U and V given
 * dH = dL/dH:
 *   dW' = A^T dH,  dW = Delta^{-1} dW',  dDelta_j = -sum_k dW'[j][k] W'[j][k] / Delta_j,
 *   G = dH W'^T + V dW^T + 1 dDelta^T,  dS = A o (G - rowsum(A o G)),
 *   dQ = scale dS U,  dV = A dW,  dU = scale sum over the batch of dS^T Q.
 * A is recomputed from Q and U (nothing is kept from the forward).
 * With d = 64 and m <= 64 the contractions run on the tensor cores (tcgen05: bf16 operands,
 * fp32 accumulators; A, W', dW and dS enter as hi + lo bf16 pairs), one CTA per slice; with
 * d = 128 and m <= 128, or d = 64 and 64 < m <= 128, also on the tensor cores, as a first pass
 * over runs of tiles, a per-slice reduce, a second pass and the dU sum (the split into runs
 * depends on the shape alone); otherwise on CUDA-core fp32 FMA.
 *
 * Inputs Q, V, dH: [B][heads][n][d]; U: [heads][m][d].  Outputs dQ, dV: [B][heads][n][d];
 * dU: [heads][m][d] (the sum over the batch entries, which share the anchors).  Device
 * pointers, 16-byte aligned, caller-owned; no output may overlap an input or another output
 * (ANCHOR_ATTN_ERR_ALIAS).  B or n = 0: dU is set to zero (dQ, dV are empty); heads = 0:
 * nothing to do.  Shapes as for the forward; anchor counts whose fp32 summaries (2 m d
 * floats) and tiles do not fit one CTA's shared memory return ANCHOR_ATTN_ERR_UNSUPPORTED
 * (for fp32: d = 16 with m > about 900, d = 32 with m > about 480).  One workspace from
 * cudaMallocAsync on `stream` per call, released on the same stream; two kernel launches
 * (four on the two-pass tensor-core path).
 * Results are bit-identical from run to run; a bounded wait that gives up is reported by
 * anchor_attn_device_error (bit 1 on the CUDA-core path, bit 0 on the tensor-core paths).
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_backward(const void *Q, const void *U, const void *V,
                                                          const void *dH, void *dQ, void *dU, void *dV, int B,
                                                          int heads, int n, int m, int d, float scale, void *stream);

/* fp32 backward: float in, float out, same layout, shapes and errors as anchor_attn_backward. */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_backward_f32(const float *Q, const float *U, const float *V,
                                                              const float *dH, float *dQ, float *dU, float *dV,
                                                              int B, int heads, int n, int m, int d, float scale,
                                                              void *stream);

/*
 * Masked (causal) variant of anchor_attn_forward: the anchors' summaries seen by token i
 * include only tokens j <= i, so that no token draws on a later one (one of the inferences of
 * the pith.science verdict on arXiv 2505.16463: A can be masked against later tokens without
 * giving up the O(mn) cost):
 *   Delta^(i)_l = sum_{j<=i} A[j][l],  W^(i)_l = sum_{j<=i} A[j][l] v_j,
 *   H[i] = sum_l A[i][l] W^(i)_l / Delta^(i)_l   (0 for an anchor with Delta^(i)_l = 0).
 * The last row equals anchor_attn_forward's last row.  Same layout, shapes, arguments and
 * errors as anchor_attn_forward; bf16 in and out.  With d = 64 and m <= 64, d = 64 and
 * 64 < m <= 128, or d = 128 and m <= 128 it runs on the tensor cores (bf16 operands, fp32
 * accumulators; one CTA per slice walks its tiles in order, the running sums inside a tile
 * taken as an MMA with a lower-triangular ones matrix; no workspace); otherwise fp32 CUDA-core
 * arithmetic (a chunked scan over the tokens, one launch,
 * one workspace from cudaMallocAsync on `stream`), where shapes whose tiles do not fit one
 * CTA's shared memory return ANCHOR_ATTN_ERR_UNSUPPORTED.  Results are bit-identical from run
 * to run; a bounded wait that gives up is reported by anchor_attn_device_error (bit 0 on the
 * tensor-core path, bit 1 on the CUDA-core path).
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_causal_forward(const void *Q, const void *U, const void *V, void *H,
                                                                int B, int heads, int n, int m, int d, float scale,
                                                                void *stream);

/* fp32 causal variant (same layout and errors). */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_causal_forward_f32(const float *Q, const float *U, const float *V,
                                                                    float *H, int B, int heads, int n, int m, int d,
                                                                    float scale, void *stream);

/*
 * Approximation-error diagnostic (the skeptic's concrete test in the pith.science verdict on
 * arXiv 2505.16463: compare the anchor construction with full softmax attention when the
 * anchors are rows of the keys).
 *
 * anchor_attn_full_forward: full softmax attention, the quadratic construction the anchors
 * approximate, H[i] = sum_j softmax over j of (scale q_i . k_j) v_j.  Q, V, H: [B][heads][n][d];
 * K: [heads][n][d], one key matrix per head shared by the batch (as the anchors U are).
 * bf16 in and out, fp32 CUDA-core arithmetic; an online softmax over 64-key tiles, so any n
 * runs; B * heads <= 65535.  d in {16, 32, 64, 128}.  H may not overlap Q, K or V.  No
 * workspace.  Meant for the diagnostic, not as a fast attention.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_full_forward(const void *Q, const void *K, const void *V, void *H,
                                                              int B, int heads, int n, int d, float scale,
                                                              void *stream);

/* fp32 full attention (same layout and errors). */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_full_forward_f32(const float *Q, const float *K, const float *V,
                                                                  float *H, int B, int heads, int n, int d,
                                                                  float scale, void *stream);

/*
 * err[b * heads + h] = ||Href[b][h] - H[b][h]||_F / ||Href[b][h]||_F (0 where Href is all
 * zero), for [B][heads][n][d] tensors of dtype 0 = bf16 or 1 = fp32; err is a device array of
 * B * heads floats.  fp32 sums of squares in a fixed order.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_relative_error(const void *Href, const void *H, float *err, int B,
                                                                int heads, int n, int d, int dtype, void *stream);

/*
 * Block front end: an AnchorFormer layer puts the anchor attention where a ViT block has its
 * self-attention, so the per-head queries and values are projections of the token embeddings
 * (pith.science verdict on arXiv 2505.16463, "key_machinery" and the referee summary of
 * Eq. 11/12; the arXiv abstract, where the anchors are weights of a trainable layer):
 *
 *   Q[b][h][i][k] = sum_c X[b][i][c] Wq[h][k][c],   V[b][h][i][k] = sum_c X[b][i][c] Wv[h][k][c]
 *   H[b][h] = anchor_attn_forward of (Q[b][h], U[h], V[b][h])
 *
 * computed in one kernel: the projections run on the tensor cores into tensor memory and are
 * used from there (rounded to bf16 operands), so X is read once and Q, V never reach global
 * memory.  Layout: X [B][n][dm]; Wq, Wv [heads][d][dm] (each head's rows of the projection
 * matrices, i.e. a [heads*d][dm] weight); U [heads][m][d]; H [B][heads][n][d]; all bf16,
 * device pointers, 16-byte aligned, caller-owned.  No bias (the pages give none).
 * Shapes: d = 64, 1 <= m <= 64, 1 <= n <= 256 (a ViT classification block: 196 patches and
 * a class token), dm a positive multiple of 64; B, heads >= 0 (zero, or n = 0, is a no-op);
 * anything else returns ANCHOR_ATTN_ERR_UNSUPPORTED.  H may not overlap X, Wq, Wv or U
 * (ANCHOR_ATTN_ERR_ALIAS).  No workspace; one launch; results are bit-identical from run to
 * run.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_block_forward(const void *X, const void *Wq, const void *Wv,
                                                               const void *U, void *H, int B, int heads, int n, int m,
                                                               int d, int dm, float scale, void *stream);

/*
 * Allocation-free variant of anchor_attn_forward (bf16 in and out, same layout, shapes and
 * errors).  The paper has no counterpart to this call: it exists for callers that may not
 * allocate device memory while they run - e.g. a plugin's enqueue step inside an inference
 * engine that owns all device memory, or a loop with a fixed memory budget - and so cannot
 * use anchor_attn_forward, which takes a workspace with cudaMallocAsync on every call.
 *
 * It always runs the chunked CUDA-core kernel (fp32 FMA, fixed-order reduction), whose
 * workspace lives in a fixed array compiled into the library:
 *   - limit: anchor_attn_static_scratch_bytes() (16 MiB); a problem needing more returns
 *     ANCHOR_ATTN_ERR_SCRATCH_LIMIT before anything is launched.  It needs
 *     roundup(4 * (32 + 2 * B * heads), 256) + 4 * B * heads * (ceil(n / 512) * (m * d + m) + m * d)
 *     bytes (a header of counters and flags, the chunk partials, W').
 *   - the array exists on every GPU that loads the library, until the process exits;
 *   - the first call on a device (and the first after the device's context changed, e.g.
 *     after cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture;
 *   - every call shares the array and it keeps the last call's contents; each call clears
 *     the header on its stream (cudaMemsetAsync, no allocation); calls whose kernels overlap
 *     on the GPU (other streams or host threads) race on it and must be serialised by the
 *     caller.
 * Calls no cudaMalloc, cudaMallocAsync, cudaFree or allocating library routine.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_forward_static_scratch(const void *Q, const void *U,
                                                                        const void *V, void *H, int B,
                                                                        int heads, int n, int m, int d,
                                                                        float scale, void *stream);

/* Size in bytes of the fixed scratch array behind anchor_attn_forward_static_scratch. */
ANCHOR_ATTN_API size_t anchor_attn_static_scratch_bytes(void);

/* Static description of what one call with these arguments launches (no GPU access).  A shape
 * that no variant can run returns ANCHOR_ATTN_ERR_UNSUPPORTED, as the forward would. */
typedef struct {
    int variant;              /* ANCHOR_ATTN_VARIANT_*                                  */
    int kernels_per_call;     /* kernel launches one call makes                        */
    int splits;               /* token chunks (CTAs) per slice whose partials are reduced */
    int flags;                /* ANCHOR_ATTN_PLAN_* (tensor-core variant)               */
    size_t workspace_bytes;   /* device workspace one call allocates (0 if none)       */
} anchor_attn_plan_t;

enum {
    ANCHOR_ATTN_PLAN_STORED_A = 1 /* pass 2 reads the A tiles pass 1 stored (else recomputes A) */
};

enum {
    ANCHOR_ATTN_VARIANT_EMPTY = 0,        /* nothing to do                                   */
    ANCHOR_ATTN_VARIANT_SIMT_SLICE = 1,   /* one CTA per slice, CUDA-core FMA                */
    ANCHOR_ATTN_VARIANT_SIMT_SPLIT = 2,   /* token chunks + fixed-order reduction, FMA       */
    ANCHOR_ATTN_VARIANT_UMMA = 3,         /* tcgen05 tensor-core path, persistent CTAs       */
    ANCHOR_ATTN_VARIANT_STREAM = 4,       /* tcgen05 tensor-core path, one CTA per slice     */
    ANCHOR_ATTN_VARIANT_SPLIT_TC = 5,     /* tcgen05, the tile list cut over 152 CTAs        */
    ANCHOR_ATTN_VARIANT_SHORT_TC = 6      /* tcgen05, one CTA per short slice, two per SM    */
};

/* dtype: 0 = bf16 (anchor_attn_forward), 1 = fp32 (anchor_attn_forward_f32).  The plan is
 * the one a call with a positive scale makes: bf16 with d = 64, 32 <= m <= 64 and n <= 256
 * runs one CTA per slice with the slice's tiles in shared memory (any scale); with n > 512 it runs
 * a slice-streaming tensor-core variant (any scale): one CTA per slice when there are at most
 * 152 slices (with at most 38 slices of many tiles, a thread-block cluster of 2 to 8 CTAs per
 * slice, the CTAs' partial sums added in rank order; `splits` = CTAs per slice, chosen from the
 * shape alone), else the slices' 128-token tiles cut into 152 contiguous ranges, one per CTA,
 * all resident at once (a device that cannot hold 152 such CTAs runs one CTA per slice
 * instead, in another summation order); otherwise the persistent tensor-core variant takes
 * bf16, d in {64, 128}, 32 <= m <= 128 and scale > 0 (a non-positive scale runs a CUDA-core
 * variant). */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_query_plan(int dtype, int B, int heads, int n, int m, int d,
                                            anchor_attn_plan_t *plan);

/*
 * Failure detection for the tensor-core variant.  Its kernel never waits without a bound:
 * a wait on the tensor-memory pipeline or on another CTA's reduction gives up after 2 s,
 * sets a bit in a device-wide error word, waits (again bounded) for the copies and MMAs it
 * has already issued, frees its tensor memory and leaves, so the context stays usable.  The
 * output of such a call is incomplete.  This call synchronises the device, copies that word
 * to *code and clears it (bit 0: a pipeline wait timed out, bit 1: a wait for a slice's
 * reduction timed out, bit 2: a wait for issued work on the way out timed out; 0: no failure
 * since the last read).  Returns ANCHOR_ATTN_ERR_CUDA if the copy fails.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_device_error(unsigned *code);

/*
 * FOR TESTS OF THE FAILURE DETECTION ONLY - not part of the forward's interface.  Runs the
 * tensor-core variant of anchor_attn_forward (ANCHOR_ATTN_ERR_UNSUPPORTED if the shape would
 * run another variant) with:
 *   hold_slice      >= 0: the reduction of that (batch, head) slice never publishes its W',
 *                   so every wait for it runs out (-1: no slice is held);
 *   wait_ns         the limit of a wait on another CTA's reduction, in ns (> 0; the
 *                   forward uses 2e9);
 *   force_recompute nonzero: pass 2 recomputes A from Q even where the stored-A plan
 *                   would run (same chunks, same result bits).
 * With a held slice the call's H is incomplete and anchor_attn_device_error reports bit 1.
 */
ANCHOR_ATTN_API anchor_attn_status_t anchor_attn_test_forward(const void *Q, const void *U, const void *V, void *H,
                                                              int B, int heads, int n, int m, int d, float scale,
                                                              int hold_slice, unsigned long long wait_ns,
                                                              int force_recompute, void *stream);

/* Human-readable name of a status code (static storage). */
ANCHOR_ATTN_API const char *anchor_attn_status_string(anchor_attn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ANCHOR_ATTN_H */

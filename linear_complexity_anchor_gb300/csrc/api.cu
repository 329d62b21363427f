// C ABI of the anchor-attention forward: argument checks, variant choice, workspace, launch.
// The operation and the argument contract are documented in include/anchor_attn.h.
#include "anchor_attn.h"
#include "common.cuh"

#include <math.h>
#include <stdlib.h>

namespace anchor {

namespace {
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
}  // namespace

anchor_attn_status_t check_shape(int B, int heads, int n, int m, int d) {
    if (B < 0 || heads < 0 || n < 0 || m < 1 || d < 1) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (!supported_d(d) || (long long)m * d > 16384) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    const long long slices = (long long)B * heads;
    // element counts must fit in 63 bits, and the work items of a call (slices x 64-token
    // blocks, and a little more) in 2^31 - 1
    if (slices > 0 && n > 0) {
        if ((long long)n * d > (1LL << 62) / slices) return ANCHOR_ATTN_ERR_INVALID_ARG;
        if (slices * ((n + 63) / 64 + (n + anchor::kSimtChunk - 1) / anchor::kSimtChunk) > 0x7fffffffLL)
            return ANCHOR_ATTN_ERR_UNSUPPORTED;
    }
    return ANCHOR_ATTN_OK;
}

anchor_attn_status_t check_problem(const Problem &p) {
    anchor_attn_status_t st = check_shape(p.B, p.heads, p.n, p.m, p.d);
    if (st != ANCHOR_ATTN_OK) return st;
    if (!isfinite(p.scale)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (p.slices() == 0 || p.n == 0) return ANCHOR_ATTN_OK;
    if (!p.Q || !p.U || !p.V || !p.H) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (!aligned16(p.Q) || !aligned16(p.U) || !aligned16(p.V) || !aligned16(p.H))
        return ANCHOR_ATTN_ERR_INVALID_ARG;
    const size_t es = p.f32 ? 4 : 2;
    const size_t xbytes = (size_t)p.slices() * p.n * p.d * es;
    const size_t ubytes = (size_t)p.heads * p.m * p.d * es;
    if (overlaps(p.H, xbytes, p.Q, xbytes) || overlaps(p.H, xbytes, p.V, xbytes) ||
        overlaps(p.H, xbytes, p.U, ubytes))
        return ANCHOR_ATTN_ERR_ALIAS;
    return ANCHOR_ATTN_OK;
}

}  // namespace anchor

namespace {

using anchor::Problem;
using anchor::check_shape;

struct Plan {
    int variant = ANCHOR_ATTN_VARIANT_EMPTY;
    int kernels = 0;
    int splits = 0;
    int flags = 0;
    size_t workspace = 0;
};

// bf16 problems with d = 64 and 32 <= m <= 64 whose slices are long (n > 512) stream each slice
// through one CTA; with more slices than kPlanSMs (a second wave of CTAs) the slices' tiles are
// cut into kPlanSMs contiguous ranges instead, one per resident CTA.  Short slices go to the
// persistent tensor-core variant, which packs several into one CTA.
bool long_plan(const Problem &p) { return anchor::split_supported(p) && p.m >= 32 && p.n > 512; }

Plan make_plan(const Problem &p) {
    Plan pl;
    if (p.slices() == 0 || p.n == 0) return pl;
    if (anchor::short_supported(p) && p.m >= 32 && p.slices() <= 0x7fffffffLL) {
        pl.variant = ANCHOR_ATTN_VARIANT_SHORT_TC;
        pl.kernels = 1;
        pl.splits = 1;
        return pl;
    }
    if (long_plan(p) && p.slices() <= 0x7fffffffLL) {
        const bool split = p.slices() > anchor::kPlanSMs;
        pl.variant = split ? ANCHOR_ATTN_VARIANT_SPLIT_TC : ANCHOR_ATTN_VARIANT_STREAM;
        pl.kernels = 1;
        pl.splits = 0;  // split: ranges of the tile list, not chunks of each slice
        if (!split) pl.splits = anchor::stream_cluster(p);  // stream: CTAs per slice
        pl.flags = ANCHOR_ATTN_PLAN_STORED_A;
        pl.workspace = split ? anchor::split_workspace(p) : anchor::stream_workspace(p);
        return pl;
    }
    if (anchor::umma_supported(p)) {
        const anchor::UmmaPlan u = anchor::umma_plan(p);
        pl.variant = ANCHOR_ATTN_VARIANT_UMMA;
        pl.kernels = 1;
        pl.splits = u.C1;
        pl.flags = u.store_a ? ANCHOR_ATTN_PLAN_STORED_A : 0;
        pl.workspace = u.workspace_bytes;
        return pl;
    }
    if (anchor::simt_full_fits(p)) {
        pl.variant = ANCHOR_ATTN_VARIANT_SIMT_SLICE;
        pl.kernels = 1;
        pl.splits = 1;
        return pl;
    }
    if (!anchor::simt_chunk_fits(p)) return pl;  // variant EMPTY with work to do: unsupported
    pl.variant = ANCHOR_ATTN_VARIANT_SIMT_SPLIT;
    pl.kernels = 1;
    pl.splits = (p.n + anchor::kSimtChunk - 1) / anchor::kSimtChunk;
    pl.workspace = anchor::simt_chunk_layout(p).total_bytes;
    return pl;
}

// test: options of the failure-detection test entry (NULL for the product entries)
struct TestRun {
    anchor::UmmaOptions opt;
    bool force_recompute;
};

anchor_attn_status_t run(const Problem &p, void *stream_v, const TestRun *test = nullptr) {
    const anchor_attn_status_t st = anchor::check_problem(p);
    if (st != ANCHOR_ATTN_OK) return st;
    if (p.slices() == 0 || p.n == 0) return ANCHOR_ATTN_OK;

    cudaStream_t stream = (cudaStream_t)stream_v;
    Plan pl = make_plan(p);
    if (test) {  // the failure-detection test entry always runs the persistent tensor-core variant
        if (!anchor::umma_supported(p)) return ANCHOR_ATTN_ERR_UNSUPPORTED;
        pl.variant = ANCHOR_ATTN_VARIANT_UMMA;
    }
    cudaError_t e = cudaSuccess;
    switch (pl.variant) {
    case ANCHOR_ATTN_VARIANT_SIMT_SLICE:
        e = anchor::launch_simt_full(p, stream);
        break;
    case ANCHOR_ATTN_VARIANT_SIMT_SPLIT: {
        void *ws = nullptr;
        if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
        if (cudaMallocAsync(&ws, pl.workspace, stream) != cudaSuccess) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_ALLOC;
        }
        e = anchor::launch_simt_chunk(p, ws, stream);
        const cudaError_t ef = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = ef;
        break;
    }
    case ANCHOR_ATTN_VARIANT_SHORT_TC:
        e = anchor::launch_short(p, stream);
        break;
    case ANCHOR_ATTN_VARIANT_STREAM:
    case ANCHOR_ATTN_VARIANT_SPLIT_TC: {
        void *ws = nullptr;
        if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
        if (cudaMallocAsync(&ws, pl.workspace, stream) != cudaSuccess) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_ALLOC;
        }
        e = pl.variant == ANCHOR_ATTN_VARIANT_SPLIT_TC ? anchor::launch_split(p, ws, stream)
                                                        : anchor::launch_stream(p, ws, stream);
        if (e == cudaErrorCooperativeLaunchTooLarge) {  // fewer resident CTAs: one CTA per slice
            cudaGetLastError();
            e = anchor::launch_stream(p, ws, stream);
        }
        const cudaError_t ef = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = ef;
        break;
    }
    case ANCHOR_ATTN_VARIANT_UMMA: {
        const anchor::UmmaPlan u = anchor::umma_plan(p, test && test->force_recompute);
        void *ws = nullptr;
        if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
        if (cudaMallocAsync(&ws, u.workspace_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_ALLOC;
        }
        e = anchor::launch_umma(p, u, test ? test->opt : anchor::UmmaOptions{}, ws, stream);
        const cudaError_t ef = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = ef;
        break;
    }
    default:
        return ANCHOR_ATTN_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();  // a failed call leaves no error behind for the caller's next check
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

// The masked (causal) variant's launch, after the forward's argument checks.
anchor_attn_status_t causal_forward(const Problem &p, void *stream_v) {
    const anchor_attn_status_t st = anchor::check_problem(p);
    if (st != ANCHOR_ATTN_OK) return st;
    if (p.slices() == 0 || p.n == 0) return ANCHOR_ATTN_OK;
    cudaStream_t stream = (cudaStream_t)stream_v;
    if (anchor::causal_tc_supported(p) || anchor::causal_wide_supported(p)) {
        if (p.slices() > 0x7fffffffLL) return ANCHOR_ATTN_ERR_UNSUPPORTED;
        const cudaError_t e = anchor::causal_tc_supported(p) ? anchor::launch_causal_tc(p, stream)
                                                             : anchor::launch_causal_wide(p, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_CUDA;
        }
        return ANCHOR_ATTN_OK;
    }
    if (!anchor::causal_fits(p)) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
    if (cudaMallocAsync(&ws, anchor::causal_layout(p).total_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_ALLOC;
    }
    cudaError_t e = anchor::launch_causal(p, ws, stream);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

// Full attention's argument checks and launch (the diagnostic's reference).
anchor_attn_status_t full_forward(const anchor::FullProblem &p, void *stream_v) {
    if (p.B < 0 || p.heads < 0 || p.n < 0 || p.d < 1) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (!(p.d == 16 || p.d == 32 || p.d == 64 || p.d == 128)) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    if (!isfinite(p.scale)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const long long S = p.slices();
    if (S == 0 || p.n == 0) return ANCHOR_ATTN_OK;
    if (S > 65535 || (long long)p.n * p.d > (1LL << 62) / S) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    const void *ptrs[4] = {p.Q, p.K, p.V, p.H};
    for (const void *q : ptrs)
        if (!q || ((uintptr_t)q & 15u)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const size_t es = p.f32 ? 4 : 2;
    const size_t xbytes = (size_t)S * p.n * p.d * es, kbytes = (size_t)p.heads * p.n * p.d * es;
    if (anchor::overlaps(p.H, xbytes, p.Q, xbytes) || anchor::overlaps(p.H, xbytes, p.V, xbytes) ||
        anchor::overlaps(p.H, xbytes, p.K, kbytes))
        return ANCHOR_ATTN_ERR_ALIAS;
    const cudaError_t e = anchor::launch_full_attention(p, (cudaStream_t)stream_v);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

// The block front end's argument checks and launch.
anchor_attn_status_t block_forward(const anchor::BlockProblem &p, void *stream_v) {
    if (p.B < 0 || p.heads < 0 || p.n < 0 || p.m < 1 || p.d < 1 || p.dm < 1) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (!isfinite(p.scale)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const long long S = (long long)p.B * p.heads;
    if (S == 0 || p.n == 0) return ANCHOR_ATTN_OK;
    if (!anchor::block_supported(p) || S > 0x7fffffffLL) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    if ((long long)p.n * p.dm > (1LL << 62) / p.B || (long long)p.n * p.d > (1LL << 62) / S)
        return ANCHOR_ATTN_ERR_INVALID_ARG;
    const void *ptrs[5] = {p.X, p.Wq, p.Wv, p.U, p.H};
    for (const void *q : ptrs)
        if (!q || ((uintptr_t)q & 15u)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const size_t xbytes = (size_t)p.B * p.n * p.dm * 2, wbytes = (size_t)p.heads * p.d * p.dm * 2;
    const size_t ubytes = (size_t)p.heads * p.m * p.d * 2, hbytes = (size_t)S * p.n * p.d * 2;
    if (anchor::overlaps(p.H, hbytes, p.X, xbytes) || anchor::overlaps(p.H, hbytes, p.Wq, wbytes) ||
        anchor::overlaps(p.H, hbytes, p.Wv, wbytes) || anchor::overlaps(p.H, hbytes, p.U, ubytes))
        return ANCHOR_ATTN_ERR_ALIAS;
    const cudaError_t e = anchor::launch_block(p, (cudaStream_t)stream_v);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

// The backward's argument checks and launch (the entry points are below).
anchor_attn_status_t backward(const anchor::BwdProblem &p, void *stream_v) {
    const anchor_attn_status_t st = check_shape(p.B, p.heads, p.n, p.m, p.d);
    if (st != ANCHOR_ATTN_OK) return st;
    if (!isfinite(p.scale)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (p.heads == 0) return ANCHOR_ATTN_OK;
    cudaStream_t stream = (cudaStream_t)stream_v;
    const size_t es = p.f32 ? 4 : 2;
    const size_t ubytes = (size_t)p.heads * p.m * p.d * es;
    if (!p.dU || ((uintptr_t)p.dU & 15u)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (p.slices() == 0 || p.n == 0) {  // no token: dU is zero
        if (cudaMemsetAsync(p.dU, 0, ubytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_CUDA;
        }
        return ANCHOR_ATTN_OK;
    }
    const void *in[4] = {p.Q, p.U, p.V, p.dH};
    const void *out[3] = {p.dQ, p.dU, p.dV};
    for (const void *q : in)
        if (!q || ((uintptr_t)q & 15u)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    for (const void *q : out)
        if (!q || ((uintptr_t)q & 15u)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const size_t xbytes = (size_t)p.slices() * p.n * p.d * es;
    const size_t in_bytes[4] = {xbytes, ubytes, xbytes, xbytes};
    const size_t out_bytes[3] = {xbytes, ubytes, xbytes};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 4; ++i)
            if (anchor::overlaps(out[o], out_bytes[o], in[i], in_bytes[i])) return ANCHOR_ATTN_ERR_ALIAS;
        for (int o2 = 0; o2 < o; ++o2)
            if (anchor::overlaps(out[o], out_bytes[o], out[o2], out_bytes[o2])) return ANCHOR_ATTN_ERR_ALIAS;
    }
    const bool wide = anchor::bwd_wide_preferred(p);
    const bool tc = !wide && anchor::bwd_tc_supported(p);
    if (!tc && !wide && !anchor::bwd_fits(p)) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
    const size_t wsb = tc     ? anchor::bwd_tc_workspace(p)
                       : wide ? anchor::bwd_wide_workspace(p)
                              : anchor::bwd_layout(p).total_bytes;
    if (cudaMallocAsync(&ws, wsb, stream) != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_ALLOC;
    }
    cudaError_t e = tc     ? anchor::launch_bwd_tc(p, ws, stream)
                    : wide ? anchor::launch_bwd_wide(p, ws, stream)
                           : anchor::launch_bwd(p, ws, stream);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

}  // namespace

namespace anchor {
anchor_attn_status_t forward_problem(const Problem &p, void *stream) { return run(p, stream); }

int forward_stream_cluster(const Problem &p) {
    if (p.slices() == 0 || p.n == 0 || make_plan(p).variant != ANCHOR_ATTN_VARIANT_STREAM) return 0;
    return stream_cluster(p);
}

}  // namespace anchor

extern "C" {

anchor_attn_status_t anchor_attn_forward(const void *Q, const void *U, const void *V, void *H, int B,
                                         int heads, int n, int m, int d, float scale, void *stream) {
    const Problem p{Q, U, V, H, B, heads, n, m, d, scale, false};
    return run(p, stream);
}

anchor_attn_status_t anchor_attn_forward_f32(const float *Q, const float *U, const float *V, float *H,
                                             int B, int heads, int n, int m, int d, float scale,
                                             void *stream) {
    const Problem p{Q, U, V, H, B, heads, n, m, d, scale, true};
    return run(p, stream);
}

anchor_attn_status_t anchor_attn_test_forward(const void *Q, const void *U, const void *V, void *H, int B,
                                              int heads, int n, int m, int d, float scale, int hold_slice,
                                              unsigned long long wait_ns, int force_recompute, void *stream) {
    if (wait_ns == 0) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const Problem p{Q, U, V, H, B, heads, n, m, d, scale, false};
    TestRun t;
    t.opt.hold_slice = hold_slice;
    t.opt.wait_ns = wait_ns;
    t.force_recompute = force_recompute != 0;
    return run(p, stream, &t);
}

anchor_attn_status_t anchor_attn_backward(const void *Q, const void *U, const void *V, const void *dH, void *dQ,
                                          void *dU, void *dV, int B, int heads, int n, int m, int d, float scale,
                                          void *stream) {
    const anchor::BwdProblem p{Q, U, V, dH, dQ, dU, dV, B, heads, n, m, d, scale, false};
    return backward(p, stream);
}

anchor_attn_status_t anchor_attn_backward_f32(const float *Q, const float *U, const float *V, const float *dH,
                                              float *dQ, float *dU, float *dV, int B, int heads, int n, int m, int d,
                                              float scale, void *stream) {
    const anchor::BwdProblem p{Q, U, V, dH, dQ, dU, dV, B, heads, n, m, d, scale, true};
    return backward(p, stream);
}

anchor_attn_status_t anchor_attn_causal_forward(const void *Q, const void *U, const void *V, void *H, int B,
                                                int heads, int n, int m, int d, float scale, void *stream) {
    return causal_forward(Problem{Q, U, V, H, B, heads, n, m, d, scale, false}, stream);
}

anchor_attn_status_t anchor_attn_causal_forward_f32(const float *Q, const float *U, const float *V, float *H, int B,
                                                    int heads, int n, int m, int d, float scale, void *stream) {
    return causal_forward(Problem{Q, U, V, H, B, heads, n, m, d, scale, true}, stream);
}

anchor_attn_status_t anchor_attn_full_forward(const void *Q, const void *K, const void *V, void *H, int B, int heads,
                                              int n, int d, float scale, void *stream) {
    return full_forward(anchor::FullProblem{Q, K, V, H, B, heads, n, d, scale, false}, stream);
}

anchor_attn_status_t anchor_attn_full_forward_f32(const float *Q, const float *K, const float *V, float *H, int B,
                                                  int heads, int n, int d, float scale, void *stream) {
    return full_forward(anchor::FullProblem{Q, K, V, H, B, heads, n, d, scale, true}, stream);
}

anchor_attn_status_t anchor_attn_block_forward(const void *X, const void *Wq, const void *Wv, const void *U, void *H,
                                               int B, int heads, int n, int m, int d, int dm, float scale,
                                               void *stream) {
    return block_forward(anchor::BlockProblem{X, Wq, Wv, U, H, B, heads, n, m, d, dm, scale}, stream);
}

anchor_attn_status_t anchor_attn_relative_error(const void *Href, const void *H, float *err, int B, int heads, int n,
                                                int d, int dtype, void *stream) {
    if ((dtype != 0 && dtype != 1) || B < 0 || heads < 0 || n < 0 || d < 1) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const long long slices = (long long)B * heads;
    if (slices == 0) return ANCHOR_ATTN_OK;
    if (slices > 0x7fffffffLL || (long long)n * d > (1LL << 62) / slices) return ANCHOR_ATTN_ERR_INVALID_ARG;
    if (!Href || !H || !err) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const cudaError_t e = anchor::launch_rel_error(Href, H, err, slices, (size_t)n * d, dtype == 1, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

anchor_attn_status_t anchor_attn_query_plan(int dtype, int B, int heads, int n, int m, int d,
                                            anchor_attn_plan_t *plan) {
    if (!plan || (dtype != 0 && dtype != 1)) return ANCHOR_ATTN_ERR_INVALID_ARG;
    const anchor_attn_status_t st = check_shape(B, heads, n, m, d);
    if (st != ANCHOR_ATTN_OK) return st;
    const Problem p{nullptr, nullptr, nullptr, nullptr, B, heads, n, m, d, 1.f, dtype == 1};
    const Plan pl = make_plan(p);
    if (pl.variant == ANCHOR_ATTN_VARIANT_EMPTY && p.slices() > 0 && n > 0) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    plan->variant = pl.variant;
    plan->kernels_per_call = pl.kernels;
    plan->splits = pl.splits;
    plan->flags = pl.flags;
    plan->workspace_bytes = pl.workspace;
    return ANCHOR_ATTN_OK;
}

anchor_attn_status_t anchor_attn_device_error(unsigned *code) {
    if (!code) return ANCHOR_ATTN_ERR_INVALID_ARG;
    unsigned a = 0, b = 0, c = 0, e = 0, f = 0, g = 0, k = 0, l = 0, q = 0, r = 0, w = 0;
    if (cudaDeviceSynchronize() != cudaSuccess || anchor::umma_read_and_clear_error(&a) != cudaSuccess ||
        anchor::simt_read_and_clear_error(&b) != cudaSuccess || anchor::bwd_read_and_clear_error(&c) != cudaSuccess ||
        anchor::causal_read_and_clear_error(&e) != cudaSuccess || anchor::block_read_and_clear_error(&f) != cudaSuccess ||
        anchor::bwd_tc_read_and_clear_error(&g) != cudaSuccess || anchor::causal_tc_read_and_clear_error(&k) != cudaSuccess ||
        anchor::stream_read_and_clear_error(&l) != cudaSuccess || anchor::split_read_and_clear_error(&q) != cudaSuccess ||
        anchor::causal_wide_read_and_clear_error(&r) != cudaSuccess ||
        anchor::bwd_wide_read_and_clear_error(&w) != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    *code = a | b | c | e | f | g | k | l | q | r | w;
    return ANCHOR_ATTN_OK;
}

const char *anchor_attn_status_string(anchor_attn_status_t s) {
    switch (s) {
    case ANCHOR_ATTN_OK: return "ok";
    case ANCHOR_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ANCHOR_ATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case ANCHOR_ATTN_ERR_ALIAS: return "output overlaps an input";
    case ANCHOR_ATTN_ERR_ALLOC: return "workspace allocation failed";
    case ANCHOR_ATTN_ERR_CUDA: return "CUDA error";
    case ANCHOR_ATTN_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch array";
    }
    return "unknown status";
}

}  // extern "C"

// Allocation-free entry point: the chunked CUDA-core kernel of the forward, with its
// workspace in a fixed array compiled into the library instead of memory taken with
// cudaMallocAsync.
//
// Who needs it: code that is not allowed to allocate device memory while it runs - a
// plugin's enqueue step inside an inference engine that owns every byte of device memory,
// or a latency-critical loop whose memory budget is fixed up front - and therefore cannot
// use anchor_attn_forward, whose chunked and tensor-core variants allocate a workspace on
// every call.
//
// The array below is part of the module: every GPU on which the library is loaded holds
// it (kStaticScratchBytes) until the process exits.  All calls share it and it keeps the
// previous call's contents; the part that must start at zero (the work ticket, arrival
// counters and ready flags) is cleared by each call with cudaMemsetAsync on the caller's
// stream, which allocates nothing.  Two calls whose kernels overlap on the GPU - on
// different streams, or from different host threads - race on it: serialise them.
#include "anchor_attn.h"
#include "common.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch.  In host code the array's name is a host-side
// stand-in, not a device address: it is translated with cudaGetSymbolAddress while the
// device is current.  The address belongs to the module loaded in one CUDA context, so it is
// kept per device together with the identity of the context it was taken in, and taken
// again when the current context is another one (after cudaDeviceReset, say).
constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id = 0;  // 0: nothing cached
    void *ptr = nullptr;
};
std::mutex g_mu;
Cached g_cache[kMaxDevices];

// identity of the calling thread's current context (0 if the driver cannot say)
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
        cudaGetLastError();
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

anchor_attn_status_t scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    // 0 when no context is current yet: the address is then taken (which makes the primary
    // context current) and taken once more on the next call, under the context's identity
    const unsigned long long id = current_context_id();
    Cached &c = g_cache[dev];
    if (id == 0 || c.ctx_id != id) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_CUDA;
        }
        c.ptr = ptr;
        c.ctx_id = id;
    }
    *out = c.ptr;
    return ANCHOR_ATTN_OK;
}

}  // namespace

extern "C" {

anchor_attn_status_t anchor_attn_forward_static_scratch(const void *Q, const void *U, const void *V, void *H,
                                                        int B, int heads, int n, int m, int d, float scale,
                                                        void *stream) {
    const anchor::Problem p{Q, U, V, H, B, heads, n, m, d, scale, false};
    const anchor_attn_status_t st = anchor::check_problem(p);
    if (st != ANCHOR_ATTN_OK) return st;
    if (p.slices() == 0 || p.n == 0) return ANCHOR_ATTN_OK;
    if (!anchor::simt_chunk_fits(p)) return ANCHOR_ATTN_ERR_UNSUPPORTED;
    if (anchor::simt_chunk_layout(p).total_bytes > kStaticScratchBytes) return ANCHOR_ATTN_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const anchor_attn_status_t s2 = scratch_for_current_device(&scratch);
    if (s2 != ANCHOR_ATTN_OK) return s2;
    const cudaError_t e = anchor::launch_simt_chunk(p, scratch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

size_t anchor_attn_static_scratch_bytes(void) { return kStaticScratchBytes; }

}  // extern "C"

// Allocation-free entry point: the token-chunk (split) CUDA-core variant of the forward,
// with its workspace in a fixed array compiled into the library instead of memory taken
// with cudaMallocAsync.
//
// Who needs it: code that is not allowed to allocate device memory while it runs - a
// plugin's enqueue step inside an inference engine that owns every byte of device memory,
// or a latency-critical loop whose memory budget is fixed up front - and therefore cannot
// use anchor_attn_forward, whose token-chunk and tensor-core variants allocate a workspace
// on every call.
//
// The array below is part of the module: every GPU on which the library is loaded holds
// it (kStaticScratchBytes) until the process exits.  All calls share it and it keeps the
// previous call's contents; nothing in it needs to start at zero (every partial is written
// before it is read).  Two calls whose kernels overlap on the GPU - on different streams,
// or from different host threads - race on it: serialise them.
#include "anchor_attn.h"
#include "common.cuh"

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device.  In host code the array's name is a
// host-side stand-in, not a device address, so it is translated once per device with
// cudaGetSymbolAddress while that device is current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

anchor_attn_status_t scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ANCHOR_ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return ANCHOR_ATTN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
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
    const int splits = (n + anchor::kSimtChunk - 1) / anchor::kSimtChunk;
    if (anchor::simt_split_workspace_bytes(p, splits) > kStaticScratchBytes) return ANCHOR_ATTN_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const anchor_attn_status_t s2 = scratch_for_current_device(&scratch);
    if (s2 != ANCHOR_ATTN_OK) return s2;
    const cudaError_t e = anchor::launch_simt_split(p, splits, static_cast<float *>(scratch),
                                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ANCHOR_ATTN_OK : ANCHOR_ATTN_ERR_CUDA;
}

size_t anchor_attn_static_scratch_bytes(void) { return kStaticScratchBytes; }

}  // extern "C"

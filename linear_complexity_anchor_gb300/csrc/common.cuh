// Shared device helpers and the internal launch interface of the anchor-attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

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
    long long slices() const { return (long long)B * heads; }
};

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
size_t simt_slice_smem_bytes(int n, int m, int d);
cudaError_t launch_simt_slice(const Problem &p, cudaStream_t stream);

constexpr int kSimtTile = 32;        // tokens per tile in the split variant
constexpr int kSimtChunk = 512;      // tokens per split (chunk) in the split variant
size_t simt_split_smem_bytes(int m, int d);
size_t simt_split_workspace_bytes(const Problem &p, int splits);
cudaError_t launch_simt_split(const Problem &p, int splits, float *workspace, cudaStream_t stream);

}  // namespace anchor

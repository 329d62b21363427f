// Two tensor-memory columns of a warp's 32 lanes to / from two registers of each lane: the
// kernels whose row warps split a row's columns in two halves exchange per-row pairs (a
// maximum and a sum) through columns that each half has already read.  The same waits and
// fences as the wider forms in ptx.cuh apply.
#pragma once

#include <stdint.h>

namespace anchor {
namespace ptx {

__device__ __forceinline__ void tmem_st2(uint32_t taddr, float a, float b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(__float_as_uint(a)),
                 "r"(__float_as_uint(b))
                 : "memory");
}
__device__ __forceinline__ float2 tmem_ld2(uint32_t taddr) {
    uint32_t x, y;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(taddr));
    return make_float2(__uint_as_float(x), __uint_as_float(y));
}

}  // namespace ptx
}  // namespace anchor

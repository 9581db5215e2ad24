// Shared device helpers and the internal launcher interface of the dflash
// library.  Nothing here is part of the C ABI (include/dflash.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

typedef __nv_bfloat16 bf16;

// ---- element conversion ----------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---- reductions ------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024).  `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < nw) ? red[lane] : 0.f;
    return warp_sum(t);
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Argmax key: value first, then the LOWEST index wins among equal values.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
    return ((unsigned long long)f32_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long k) {
    return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}

// Device error word bits (set with atomicOr, read by the host at sync points).
enum : uint32_t {
    ERR_TOKEN_RANGE = 1u,
    ERR_POSITION_RANGE = 2u,
    ERR_TIMEOUT = 4u
};

// ---- programmatic dependent launch -------------------------------------------
// Every kernel of the round may be launched so that it starts while the kernel
// before it is still running.  pdl_wait() blocks until that kernel has finished
// and its writes are visible; each kernel calls it in every thread before it
// reads anything an earlier kernel wrote (and before it can exit), so kernel
// completion stays ordered.  pdl_trigger() lets the next kernel start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- paged KV addressing ---------------------------------------------------
// A cache layer is [num_pages][H_kv][page_tokens][hd]; page_table[seq * pages_per_seq + i]
// gives the physical page of the seq's i-th block of page_tokens positions.
struct KVLayout {
    int page_tokens;      // tokens per page (power of two)
    int page_shift;       // log2(page_tokens)
    int pages_per_seq;
    int n_kv_heads;
    int head_dim;
    long long layer_stride;  // elements per layer of one cache (K or V)
};

__device__ __forceinline__ long long kv_offset(const KVLayout& L, const int* page_table, int seq, int pos,
                                               int kvh) {
    const int page = page_table[seq * L.pages_per_seq + (pos >> L.page_shift)];
    const int slot = pos & (L.page_tokens - 1);
    return (((long long)page * L.n_kv_heads + kvh) * L.page_tokens + slot) * L.head_dim;
}

}  // namespace dfl

// kda_common.cuh -- shared device helpers of libkda.so (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Status word at offset 0 of every workspace (16 bytes; the first 256 bytes
// of a workspace are reserved for it).
struct StatusWord {
    uint32_t code;
    uint32_t site;
    unsigned long long info;
};
constexpr size_t kHeaderBytes = 256;

// g_min of the lower-bounded log-decay (dev.to page, "The Sequence
// Bottleneck", the gate equation and the paragraph after it).
constexpr float kGMin = -5.0f;
// Bound on the cumulative log-decay of one 16-token tile (same paragraph).
constexpr float kTileDecayBound = -80.0f;
constexpr int kTile = 16;

// Optional timing hook: records caller-created CUDA events on the launch stream
// before the first kernel and after every kernel of one call.
struct EventRec {
    cudaEvent_t *ev = nullptr;
    int cap = 0;
    int used = 0;
    // records the next event on `s`; each kernel is bracketed by two marks on its own stream
    void mark(cudaStream_t s) {
        if (ev && used < cap) cudaEventRecord(ev[used++], s);
    }
};

__device__ __forceinline__ void report(StatusWord *st, uint32_t code, long long info,
                                       uint32_t site = 0) {
    if (st == nullptr) return;
    if (atomicCAS(&st->code, 0u, code) == 0u) {
        st->site = site;
        atomicExch(&st->info, (unsigned long long)info);
    }
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// The gate: g = g_min * Sigmoid(expA * z) with Sigmoid(x) = 1 / (1 + exp(-x)).
// expA = exp(A_h) is computed once per head by the caller.  Large positive
// arguments give g = g_min, large negative ones g = -0; NaN propagates.
__device__ __forceinline__ float gate(float z, float expA) {
    return kGMin / (1.0f + expf(-expA * z));
}

// A cumulative decay passes the tile check when finite and inside the
// closed interval [-80, 0] (floating-point rounding can reach either end of
// the open interval the page states).
__device__ __forceinline__ bool decay_ok(float G) {
    return G >= kTileDecayBound && G <= 0.0f;  // false for NaN
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace kda

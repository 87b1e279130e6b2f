// kda_common.cuh -- small helpers shared by the KDA kernels (device side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;   // tokens per chunk of the chunk-parallel prefill

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Device status word at the start of the prefill workspace.
struct DeviceHeader {
    int32_t status;        // kda_status recorded by the device
    int32_t total_chunks;  // sum over sequences of ceil(len / kChunk)
    int32_t pad[62];       // keeps the chunk table 256-byte aligned (pad[0..1]: cu_seqlens of a
                           // single sequence; pad[kHdrSlowChunk]: see below)
};
// pad[kHdrSlowChunk] is cleared by the sequence-table kernel and set to 1 by
// the tensor-core intra-chunk kernel when some chunk's cumulative decay is
// too strong for its factorised products (it then takes its slow path).  The
// tensor-core backward reads it to hand such calls to the CUDA-core backward.
constexpr int kHdrSlowChunk = 8;

__device__ __forceinline__ void record_status(DeviceHeader* hdr, int code) {
    atomicCAS(&hdr->status, (int)KDA_OK, code);
}

// Index of the sequence that owns global chunk `c`, given the exclusive prefix
// of chunk counts chunk_first[0..N] (chunk_first[N] = total chunks).
__device__ __forceinline__ int chunk_owner(const int32_t* chunk_first, int N, int c) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_first[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace kda

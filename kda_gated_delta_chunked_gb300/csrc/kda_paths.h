// kda_paths.h -- host-side entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

enum PrefillPath { kPathSimt = 0, kPathTensorCore = 1 };

// Which prefill implementation runs for a dtype, head size and desc flags.
int choose_prefill_path(int dtype, int d, int flags);
// Bytes of workspace per (chunk, head) record for a path.
size_t prefill_record_bytes(int path, int d);
// Bytes of path-specific scratch after the records.
size_t prefill_extra_bytes(int path, int N, int H, int64_t T);

// Launch arguments shared by the prefill paths.
struct PrefillArgs {
    int dtype, d, N, H, chunks_ub;
    int64_t T;                   // total tokens
    const void *q, *k, *v, *la, *beta;
    int la_scalar;               // 1: la is [T, H] (one gate per token and head), else [T, H, d]
    const int32_t* cu;           // device cu_seqlens (or the workspace copy)
    const float* s0;             // initial state or nullptr
    void* out;
    float* sf;                   // final state or nullptr
    void* hdr;                   // DeviceHeader in the workspace
    const int32_t* chunk_first;  // [N+1] chunk offsets in the workspace
    void* recs;                  // per-(chunk, head) records
    void* extra;                 // path-specific scratch after the records
    cudaEvent_t* phase_events;   // optional timing events (3) or nullptr
    const int32_t* snap_slot;    // [chunks] snapshot index to write after each chunk (-1: none), or nullptr
    float* snaps;                // snapshot states [M, H, d, d] (with snap_slot)
};

cudaError_t prefill_launch(int path, const PrefillArgs& a, cudaStream_t stream);

// Reverse mode of the prefill (kda_backward.cu).
struct BackwardArgs {
    int dtype, d, N, H;
    int64_t T;
    const void *q, *k, *v, *la, *beta, *dout;
    int la_scalar;
    const int32_t* cu;
    const float *s0, *dfinal;
    float *dq, *dk, *dv, *dla, *dbeta, *ds0;
    void* hdr;
    const int32_t* chunk_first;
    float* ckpt;                 // kept states, backward_ckpt_bytes
    float* part;                 // per-tile partial sums, backward_part_bytes
    int only_if_slow;            // 1: the CUDA-core kernels run only when the header's slow-chunk
                                 //    flag is set (fallback of the tensor-core backward)
};
size_t backward_ckpt_bytes(int d, int H, int64_t chunks_ub);
size_t backward_part_bytes(int N, int d, int H, int64_t T);
cudaError_t backward_launch(const BackwardArgs& a, cudaStream_t stream);

cudaError_t decode_step_launch(int dtype, int d, const void* q, const void* k, const void* v,
                               const void* la, int la_scalar, const void* beta, float* state, void* out,
                               int N, int H, cudaStream_t stream);

// CUDA-core (fp32) prefill.
size_t simt_record_bytes(int d);
cudaError_t prefill_simt_launch(const PrefillArgs& a, cudaStream_t stream);

// Tensor-core (tcgen05) prefill: bf16 inputs, head size 128.
size_t tc_record_bytes();
size_t tc_extra_bytes(int N, int H, int64_t T);
cudaError_t prefill_tc_launch(const PrefillArgs& a, int64_t T, cudaStream_t stream);
// Tensor map of a [T, H, 128] bf16 tensor with 64-token x 64-channel boxes of
// one head, 128-byte swizzle (a canonical MN-major operand tile per box).
bool tc_make_tile_map(CUtensorMap* m, const void* base, int64_t T, int H);

// Tensor-core backward (kda_backward_tc.cu): bf16 inputs, head size 128.
size_t backward_tc_bytes(int N, int H, int64_t T, int64_t chunks_ub);
cudaError_t backward_tc_launch(const BackwardArgs& a, int64_t chunks_ub, void* region, cudaStream_t stream);

}  // namespace kda

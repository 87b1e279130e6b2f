// kda_tc_record.cuh -- layout of the per-(chunk, head) record that the
// tensor-core intra-chunk kernel writes and the inter-chunk kernels (forward
// chain, reverse chain of the backward) read.  Head size 128, chunk 64.
#pragma once

#include <stdint.h>

namespace kda {

constexpr int kTile = 16;                  // columns per tile of the O0 record image
constexpr float kTcMaxSpanLog2 = 100.f;    // the factorised chunk products hold while max_c (-g_C) <= 100 (log2)

// Record of one (chunk, head), byte offsets.  With g the running sum of
// log alpha from the chunk start and T = (I + A)^-1 Diag(beta):
struct TcRec {
    static constexpr uint32_t kA1 = 0;          // [W; Q'] = [T K~; Q~ - P T K~], 128 rows x 128 channels,
                                                //   2 channel blocks x [128 rows x 128 B], 128-byte swizzle
    static constexpr uint32_t kKE = 32768;      // K^end = K * exp(g_C - g): token-major, 2 x [64 tok x 64 ch]
    static constexpr uint32_t kU0 = 49152;      // U0 = T V: token-major, 2 x [64 tok x 64 ch], 128-byte swizzle
    static constexpr uint32_t kO0 = 65536;      // O0 = P T V: 8 tiles x [64 tokens x 16] bf16
    static constexpr uint32_t kGam = 81920;     // Gamma = exp(g_C): 128 fp32
    static constexpr uint32_t kBytes = 82432;
    static constexpr uint32_t kTileBytes = 64 * kTile * 2;
};

}  // namespace kda

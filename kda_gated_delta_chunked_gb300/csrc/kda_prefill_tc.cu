// kda_prefill_tc.cu -- chunk-parallel KDA prefill on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA), bf16 operands with fp32
// accumulation and an fp32 state.  Head size 128.
//
// The chunk algebra is the one of the CUDA-core path (kda_prefill_simt.cu):
// within a chunk of C = 64 tokens with start state S0 and g_r the running sum
// of log alpha (per key channel),
//
//   A  = Diag(beta) StrictLower(K~ K^T)      P = LowerIncl(Q~ K^T)
//   T  = (I + A)^-1 Diag(beta)
//   W  = T K~     U0 = T V     Q' = Q~ - P T K~     O0 = P T V
//   K^end = K * exp(g_C - g),  Gamma = exp(g_C)
//
// and across the chunks of a sequence, in order:
//   U = U0 - W S,   O = O0 + Q' S,   S <- Diag(Gamma) S + K^end^T U.
//
// ("Kimi Delta Attention" deep dive, section 06: matrix products inside a
// chunk, the recurrent state carried between chunks; the recurrence itself is
// that of section 03.)
//
// Kernel (a), one CTA per (chunk, head), 128 threads:
//   1. TMA loads the q, k, v, log_alpha tiles [64 tokens x 128].
//   2. Thread c owns key channel c: running sum g, then every scaled operand
//      (K~, Q~, K^ around a mid-chunk reference for the Gram products; K~ and
//      Q~ from the chunk start and V, transposed, for the second product;
//      K^end transposed for kernel b), written as bf16 in the 128-byte-swizzle
//      K-major layout the tensor core reads.
//   3. MMA-a (M=128, N=64, K=128): [K~m; Q~m] K^m^T gives the Gram block (rows
//      0..63, -> A) and the P block (rows 64..127) in one TMEM accumulator.
//   4. One recursion per row gives [T; P T] at once: Y (I + A) = [I; P], solved
//      column by column from the right, then scaled by Diag(beta).
//   5. MMA-b (M=128, N=256 then 128, K=64+64):
//        [[T, 0], [P T, -I]] x [[K~, V], [Q~, 0]] = [[W, U0], [-Q', O0]].
//   6. The records kernel (b) reads are written as ready-to-copy shared-memory
//      images: [W; Q'] and K^end^T in the swizzled K-major layout, U0 / O0 in
//      16-column tiles, Gamma.
// Chunks whose cumulative decay spans more than 2^100 inside the chunk cannot
// use the mid-reference factorisation in fp32; for those the Gram and P blocks
// are formed on CUDA cores with exp(g_i - g_j) inside the sum (never > 1).
//
// Kernel (b), one CTA per (sequence, head, 16-column tile of the state):
// a producer warp streams each chunk's record into a 3-stage shared-memory
// ring with 1-D bulk copies; four consumer warps keep their 128 x 16 slice of
// S in fp32 registers (thread i = key channel i) and per chunk issue
//   MMA1 (M=128, N=16, K=128): [W; Q'] S  -> U = U0 - W S (rows 0..63),
//                                             O = O0 + Q' S (rows 64..127)
//   MMA3 (M=128, N=16, K=64):  K^end^T U  -> S <- Gamma * S + K^end^T U
// with S and U fed back to the tensor core as bf16 operands.
//
// Every wait on an mbarrier is bounded; on timeout the kernel records
// KDA_ERR_TIMEOUT in the device status word, drains its own copies and exits.
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_paths.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

constexpr int kTcD = 128;                // head size handled here
constexpr int kTile = 16;                // state columns per CTA of kernel (b)
constexpr int kTiles = kTcD / kTile;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxSpanLog2 = 100.f;    // fast path if max_c (g_0 - g_C) <= 2^100 (log2 units)

// Record of one (chunk, head), bytes.
struct TcRec {
    static constexpr uint32_t kA1 = 0;          // [W; Q'] image: 2 K-blocks x [128 rows x 128 B]
    static constexpr uint32_t kKE = 32768;      // K^end^T image: [128 rows x 128 B]
    static constexpr uint32_t kU0 = 49152;      // U0: 8 tiles x [64 tokens x 16] bf16
    static constexpr uint32_t kO0 = 65536;      // O0: same layout
    static constexpr uint32_t kGam = 81920;     // Gamma: 128 fp32
    static constexpr uint32_t kBytes = 82432;
    static constexpr uint32_t kTileBytes = 64 * kTile * 2;
};

size_t tc_record_bytes() { return TcRec::kBytes; }

// ---------------------------------------------------------------------------
// Kernel (a)
// ---------------------------------------------------------------------------
struct SmemA {   // byte offsets from a 1024-aligned base
    static constexpr uint32_t kIn = 0;          // K, Q, LA, V tiles (TMA), 4 x 16 KB
    static constexpr uint32_t kInK = 0, kInQ = 16384, kInLA = 32768, kInV = 49152;
    static constexpr uint32_t kOpA = 65536;     // MMA-a A [K~m; Q~m], 32 KB; later At fp32 (16 KB)
    static constexpr uint32_t kOpB1 = 98304;    // MMA-a B K^m, 16 KB
    static constexpr uint32_t kOpB2 = 114688;   // MMA-b B: [K~^T; V^T] (32 KB) + Q~^T (16 KB)
    static constexpr uint32_t kKE = 163840;     // K^end^T image, 16 KB
    static constexpr uint32_t kMisc = 180224;   // beta, flags, barriers
    static constexpr uint32_t kBytes = 181248 + 1024;
    // After step 2: MMA-b A operand [[T,0],[PT,-I]] reuses the K/Q tiles (32 KB),
    // the slow path keeps g (fp32 [64][128]) in the LA/V tiles.
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

__global__ void __launch_bounds__(128, 1)
kda_tc_intra_chunk(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                   const __nv_bfloat16* __restrict__ beta, const int32_t* __restrict__ cu,
                   DeviceHeader* __restrict__ hdr, const int32_t* __restrict__ chunk_first, int N, int H,
                   uint8_t* __restrict__ recs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* s_beta = (float*)(sm + SmemA::kMisc);                 // [64]
    uint64_t* bars = (uint64_t*)(sm + SmemA::kMisc + 256);       // [0] inputs, [1] mma
    uint32_t* s_tmem = (uint32_t*)(sm + SmemA::kMisc + 512);
    int* s_flag = (int*)(sm + SmemA::kMisc + 528);                // [0] slow path, [1] abort

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (hdr->status != KDA_OK) return;
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= hdr->total_chunks) return;
    const int n = chunk_owner(chunk_first, N, c);
    const int64_t t0 = (int64_t)cu[n] + (int64_t)(c - chunk_first[n]) * kChunk;
    const int len = (int)min64(kChunk, (int64_t)cu[n + 1] - t0);
    uint8_t* rec = recs + ((size_t)c * H + h) * TcRec::kBytes;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        s_flag[0] = 0;
        s_flag[1] = 0;
        prefetch_tensormap(&tm_q); prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v); prefetch_tensormap(&tm_la);
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 4 * 16384);
        tma_load_3d(sm + SmemA::kInK, &tm_k, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + SmemA::kInQ, &tm_q, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + SmemA::kInLA, &tm_la, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + SmemA::kInV, &tm_v, 0, h, (int)t0, &bars[0]);
    }
    if (tid < kChunk) s_beta[tid] = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    if (warp == 0) { tmem_alloc(s_tmem, 256); tmem_relinquish(); }
    if (!mbar_wait(&bars[0], 0, kWaitNs)) s_flag[1] = 1;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    bool abort = s_flag[1] != 0;

    // ---- step 2a: running sum of log alpha for channel c (log2 units) ----
    const int ch = tid;                        // key channel owned by this thread
    const __nv_bfloat16* inK = (const __nv_bfloat16*)(sm + SmemA::kInK);
    const __nv_bfloat16* inQ = (const __nv_bfloat16*)(sm + SmemA::kInQ);
    const __nv_bfloat16* inL = (const __nv_bfloat16*)(sm + SmemA::kInLA);
    const __nv_bfloat16* inV = (const __nv_bfloat16*)(sm + SmemA::kInV);
    float G[kChunk];
    {
        float g = 0.f;
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const float la = r < len ? __bfloat162float(inL[r * kTcD + ch]) : 0.f;
            g = fmaf(la, kLog2e, g);
            G[r] = g;
        }
    }
    const float gm = G[31], gC = G[kChunk - 1];
    if (G[0] - gC > kMaxSpanLog2) s_flag[0] = 1;   // benign race: any writer sets 1
    __syncthreads();
    const bool slow = s_flag[0] != 0;

    // ---- step 2b: scaled operands ----
    {
        const uint32_t kb = (uint32_t)ch >> 6, kin = (uint32_t)ch & 63u;
        uint8_t* opA = sm + SmemA::kOpA + kb * 16384;
        uint8_t* opB1 = sm + SmemA::kOpB1 + kb * 8192;
        uint8_t* opB2 = sm + SmemA::kOpB2;
        uint8_t* keI = sm + SmemA::kKE;
        const float Em = exp2f(gm), ECm = exp2f(gC - gm);
        uint32_t kt[4], qt[4], vt[4], ke[4];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const bool ok = r < len;
            const float kv = ok ? __bfloat162float(inK[r * kTcD + ch]) : 0.f;
            const float qv = ok ? __bfloat162float(inQ[r * kTcD + ch]) : 0.f;
            const float vv = ok ? __bfloat162float(inV[r * kTcD + ch]) : 0.f;
            float e3, e4;
            if (!slow) {
                const float e1 = exp2f(G[r] - gm);         // 2^(g_r - g_m)
                const float e2 = exp2f(gm - G[r]);         // 2^(g_m - g_r)
                e3 = e1 * Em;                              // 2^(g_r)        <= 1
                e4 = e2 * ECm;                             // 2^(g_C - g_r)  <= 1
                *(__nv_bfloat16*)(opA + sw128_off(r, kin)) = __float2bfloat16_rn(kv * e1);
                *(__nv_bfloat16*)(opA + sw128_off(64 + r, kin)) = __float2bfloat16_rn(qv * e1);
                *(__nv_bfloat16*)(opB1 + sw128_off(r, kin)) = __float2bfloat16_rn(kv * e2);
            } else {
                e3 = exp2f(G[r]);
                e4 = exp2f(gC - G[r]);
            }
            const int w = (r & 7) >> 1;
            if ((r & 1) == 0) {
                kt[w] = pack_bf16x2(kv * e3, 0.f); qt[w] = pack_bf16x2(qv * e3, 0.f);
                vt[w] = pack_bf16x2(vv, 0.f);      ke[w] = pack_bf16x2(kv * e4, 0.f);
            } else {
                kt[w] = (kt[w] & 0xffffu) | (pack_bf16x2(0.f, kv * e3) & 0xffff0000u);
                qt[w] = (qt[w] & 0xffffu) | (pack_bf16x2(0.f, qv * e3) & 0xffff0000u);
                vt[w] = (vt[w] & 0xffffu) | (pack_bf16x2(0.f, vv) & 0xffff0000u);
                ke[w] = (ke[w] & 0xffffu) | (pack_bf16x2(0.f, kv * e4) & 0xffff0000u);
            }
            if ((r & 7) == 7) {
                const uint32_t r8 = (uint32_t)(r & ~7);
                *(uint4*)(opB2 + sw128_off(ch, r8)) = make_uint4(kt[0], kt[1], kt[2], kt[3]);
                *(uint4*)(opB2 + sw128_off(128 + ch, r8)) = make_uint4(vt[0], vt[1], vt[2], vt[3]);
                *(uint4*)(opB2 + 32768 + sw128_off(ch, r8)) = make_uint4(qt[0], qt[1], qt[2], qt[3]);
                *(uint4*)(keI + sw128_off(ch, r8)) = make_uint4(ke[0], ke[1], ke[2], ke[3]);
            }
        }
        ((float*)(rec + TcRec::kGam))[ch] = exp2f(gC);
    }
    fence_proxy_async_smem();
    __syncthreads();

    float* At = (float*)(sm + SmemA::kOpA);       // At[j][i] = A[i][j], fp32 [64][64] (after MMA-a)
    float Y[kChunk];                              // row `tid` of [X; P X], X = (I + A)^-1
    if (!slow) {
        if (tid == 0 && !abort) {
            // K^end^T image -> record (smem read by the copy engine, async)
            bulk_s2g(rec + TcRec::kKE, sm + SmemA::kKE, 16384);
            bulk_commit();
            tc_fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = ks & 3;
                mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(sm + SmemA::kOpA + kb * 16384 + kin * 32)),
                            sdesc_k_sw128(smem_u32(sm + SmemA::kOpB1 + kb * 8192 + kin * 32)), id, ks > 0);
            }
            mma_commit(&bars[1]);
        }
        if (!abort && !mbar_wait(&bars[1], 0, kWaitNs)) { s_flag[1] = 1; }
        tc_fence_after_sync();
        // D rows 0..63 (warps 0,1): Gram -> A^T; rows 64..127 (warps 2,3): P row in registers.
        float d[kChunk];
#pragma unroll
        for (int c0 = 0; c0 < kChunk; c0 += 16) {
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, c0), f);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) d[c0 + j] = f[j];
        }
        tc_fence_before_sync();
        __syncthreads();                          // everyone done with MMA-a operands
        if (warp < 2) {
            const int i = tid;                    // token row of the Gram block
            const float bi = s_beta[i];
#pragma unroll
            for (int j = 0; j < kChunk; ++j) At[j * kChunk + i] = (j < i) ? bi * d[j] : 0.f;
#pragma unroll
            for (int j = 0; j < kChunk; ++j) Y[j] = (j == i) ? 1.f : 0.f;
        } else {
            const int i = tid - 64;
#pragma unroll
            for (int j = 0; j < kChunk; ++j) Y[j] = (j <= i) ? d[j] : 0.f;
        }
    } else {
        // Slow path: g to shared memory (fp32 [64][128] over the LA/V tiles), then
        // A and P on CUDA cores with exp(g_i - g_j) inside the sums.
        float* gS = (float*)(sm + SmemA::kInLA);
#pragma unroll
        for (int r = 0; r < kChunk; ++r) gS[r * kTcD + ch] = G[r];
        if (tid == 0 && !abort) {
            bulk_s2g(rec + TcRec::kKE, sm + SmemA::kKE, 16384);
            bulk_commit();
        }
        __syncthreads();
        float* Ps = (float*)(sm + SmemA::kOpA + 16384);   // P fp32 [64][64]
        for (int e = tid; e < kChunk * kChunk; e += 128) {
            const int i = e >> 6, j = e & 63;
            float a = 0.f, p = 0.f;
            if (j <= i && i < len) {
                for (int cc = 0; cc < kTcD; ++cc) {
                    const float ek = __bfloat162float(inK[j * kTcD + cc]) *
                                     exp2f(gS[i * kTcD + cc] - gS[j * kTcD + cc]);
                    a = fmaf(__bfloat162float(inK[i * kTcD + cc]), ek, a);
                    p = fmaf(__bfloat162float(inQ[i * kTcD + cc]), ek, p);
                }
            }
            At[j * kChunk + i] = (j < i) ? s_beta[i] * a : 0.f;
            Ps[i * kChunk + j] = p;
        }
        __syncthreads();
        if (warp < 2) {
#pragma unroll
            for (int j = 0; j < kChunk; ++j) Y[j] = (j == tid) ? 1.f : 0.f;
        } else {
#pragma unroll
            for (int j = 0; j < kChunk; ++j) Y[j] = Ps[(tid - 64) * kChunk + j];
        }
    }
    __syncthreads();                              // At complete

    // ---- step 4: Y (I + A) = [I; P], columns from the right ----
    {
        const float4* At4 = (const float4*)At;
#pragma unroll
        for (int j = kChunk - 2; j >= 0; --j) {
            float acc = Y[j];
#pragma unroll
            for (int g4 = (j + 1) >> 2; g4 < kChunk / 4; ++g4) {
                const float4 a = At4[j * (kChunk / 4) + g4];
                if (4 * g4 + 0 > j) acc = fmaf(-Y[4 * g4 + 0], a.x, acc);
                if (4 * g4 + 1 > j) acc = fmaf(-Y[4 * g4 + 1], a.y, acc);
                if (4 * g4 + 2 > j) acc = fmaf(-Y[4 * g4 + 2], a.z, acc);
                if (4 * g4 + 3 > j) acc = fmaf(-Y[4 * g4 + 3], a.w, acc);
            }
            Y[j] = acc;
        }
    }
    // ---- step 5: row `tid` of [[T, 0], [P T, -I]] as the MMA-b A operand ----
    {
        uint8_t* opA2 = sm + SmemA::kInK;          // 2 K-blocks x [128 rows x 128 B] over the K/Q tiles
        const int row = tid;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = c8 * 8 + 2 * e;
                w4[e] = pack_bf16x2(Y[j] * s_beta[j], Y[j + 1] * s_beta[j + 1]);
            }
            *(uint4*)(opA2 + sw128_off(row, c8 * 8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            uint32_t z[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = c8 * 8 + 2 * e;
                const float lo = (row >= 64 && row - 64 == j) ? -1.f : 0.f;
                const float hi = (row >= 64 && row - 64 == j + 1) ? -1.f : 0.f;
                z[e] = pack_bf16x2(lo, hi);
            }
            *(uint4*)(opA2 + 16384 + sw128_off(row, c8 * 8)) = make_uint4(z[0], z[1], z[2], z[3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    abort = abort || s_flag[1] != 0;
    if (tid == 0 && !abort) {
        const uint32_t id256 = idesc_bf16(128, 256), id128 = idesc_bf16(128, 128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(sm + SmemA::kInK + ks * 32)),
                        sdesc_k_sw128(smem_u32(sm + SmemA::kOpB2 + ks * 32)), id256, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(sm + SmemA::kInK + 16384 + ks * 32)),
                        sdesc_k_sw128(smem_u32(sm + SmemA::kOpB2 + 32768 + ks * 32)), id128, 1);
        mma_commit(&bars[1]);
    }
    if (!abort && !mbar_wait(&bars[1], slow ? 0 : 1, kWaitNs)) s_flag[1] = 1;
    tc_fence_after_sync();

    // ---- step 6: epilogue.  Warps 0,1: rows 0..63 = [W | U0]; warps 2,3: rows 64..127 = [-Q' | O0].
    if (!abort) {
        const int i = (warp & 1) * 32 + lane;      // token row within the chunk
        const bool top = warp < 2;
        uint8_t* a1 = rec + TcRec::kA1;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, c0), f);
            tmem_wait_ld();
            const float sgn = top ? 1.f : -1.f;    // rows 64..127 hold -Q'
            uint32_t p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p[e] = pack_bf16x2(sgn * f[2 * e], sgn * f[2 * e + 1]);
            const int row = top ? i : 64 + i;
            const uint32_t kb = c0 >> 6, kin = c0 & 63;
            *(uint4*)(a1 + kb * 16384 + sw128_off(row, kin)) = make_uint4(p[0], p[1], p[2], p[3]);
            *(uint4*)(a1 + kb * 16384 + sw128_off(row, kin + 8)) = make_uint4(p[4], p[5], p[6], p[7]);
        }
        uint8_t* uo = rec + (top ? TcRec::kU0 : TcRec::kO0);
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 128 + t * kTile), f);
            tmem_wait_ld();
            uint32_t p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
            uint4* dst = (uint4*)(uo + t * TcRec::kTileBytes + i * (kTile * 2));
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
        }
    } else if (tid == 0) {
        record_status(hdr, KDA_ERR_TIMEOUT);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    if (tid == 0) bulk_wait_all();                // the K^end image store has read its smem
}

// ---------------------------------------------------------------------------
// Kernel (b)
// ---------------------------------------------------------------------------
constexpr int kStages = 3;
struct SmemB {
    static constexpr uint32_t kStageA1 = 0, kStageKE = 32768, kStageU0 = 49152, kStageO0 = 51200,
                              kStageGam = 53248, kStageBytes = 54272;       // 53 KB, 1024-aligned
    static constexpr uint32_t kST = kStages * kStageBytes;                 // S^T operand, 2 x 2 KB
    static constexpr uint32_t kUT = kST + 4096;                            // U^T operand, 2 KB
    static constexpr uint32_t kMisc = kUT + 2048;                          // barriers etc.
    static constexpr uint32_t kBytes = kMisc + 256 + 1024;
    static constexpr uint32_t kTx = 32768 + 16384 + 2 * TcRec::kTileBytes + 512;
};

__global__ void __launch_bounds__(160, 1)
kda_tc_inter_chunk(const int32_t* __restrict__ cu, DeviceHeader* __restrict__ hdr,
                   const int32_t* __restrict__ chunk_first, int H, const uint8_t* __restrict__ recs,
                   const float* __restrict__ initial_state, __nv_bfloat16* __restrict__ out,
                   float* __restrict__ final_state) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(sm + SmemB::kMisc);            // [kStages]
    uint64_t* empty = full + kStages;                           // [kStages]
    uint64_t* mbar1 = empty + kStages;
    uint64_t* mbar3 = mbar1 + 1;
    uint32_t* s_tmem = (uint32_t*)(mbar3 + 1);
    int* s_abort = (int*)(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (hdr->status != KDA_OK) return;
    const int nh = blockIdx.x, n = nh / H, h = nh % H;
    const int col0 = blockIdx.y * kTile;
    const int c_begin = chunk_first[n], nchunks = chunk_first[n + 1] - c_begin;
    const int64_t seq0 = cu[n], seq1 = cu[n + 1];

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(mbar1, 1);
        mbar_init(mbar3, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) { tmem_alloc(s_tmem, 32); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;

    if (warp == 4) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nchunks; ++it) {
                const int s = it % kStages;
                if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1, kWaitNs)) {
                    *(volatile int*)s_abort = 1;
                    break;
                }
                if (*(volatile int*)s_abort) break;
                const uint8_t* rec = recs + ((size_t)(c_begin + it) * H + h) * TcRec::kBytes;
                uint8_t* st = sm + s * SmemB::kStageBytes;
                mbar_arrive_expect_tx(&full[s], SmemB::kTx);
                bulk_g2s(st + SmemB::kStageA1, rec + TcRec::kA1, 32768, &full[s]);
                bulk_g2s(st + SmemB::kStageKE, rec + TcRec::kKE, 16384, &full[s]);
                bulk_g2s(st + SmemB::kStageU0, rec + TcRec::kU0 + blockIdx.y * TcRec::kTileBytes,
                         TcRec::kTileBytes, &full[s]);
                bulk_g2s(st + SmemB::kStageO0, rec + TcRec::kO0 + blockIdx.y * TcRec::kTileBytes,
                         TcRec::kTileBytes, &full[s]);
                bulk_g2s(st + SmemB::kStageGam, rec + TcRec::kGam, 512, &full[s]);
                issued = it + 1;
            }
            // Drain: every copy this warp issued has landed before the CTA may exit.
            for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
                mbar_wait(&full[it % kStages], (it / kStages) & 1, kWaitNs);
        }
    } else {
        // ---------------- consumers: thread i = key channel i ----------------
        const int i = tid;
        const size_t sbase = (size_t)nh * kTcD * kTcD + (size_t)i * kTcD + col0;
        float S[kTile];
        if (initial_state) {
            const float4* p = (const float4*)(initial_state + sbase);
#pragma unroll
            for (int q4 = 0; q4 < kTile / 4; ++q4) {
                const float4 v = p[q4];
                S[4 * q4] = v.x; S[4 * q4 + 1] = v.y; S[4 * q4 + 2] = v.z; S[4 * q4 + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kTile; ++j) S[j] = 0.f;
        }
        uint8_t* ST = sm + SmemB::kST;
        uint8_t* UT = sm + SmemB::kUT;
        auto write_ST = [&]() {
            const uint32_t kb = (uint32_t)i >> 6, kin = (uint32_t)i & 63u;
#pragma unroll
            for (int j = 0; j < kTile; ++j)
                *(__nv_bfloat16*)(ST + kb * 2048 + sw128_off(j, kin)) = __float2bfloat16_rn(S[j]);
        };
        write_ST();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        // Consumers meet only at barriers that AND a "still good" flag, so a
        // wait that timed out in any thread stops all of them together.
        bool ok = bar_and(128, true);
        const uint32_t id = idesc_bf16(128, kTile);
        for (int it = 0; it < nchunks; ++it) {
            const int s = it % kStages;
            uint8_t* st = sm + s * SmemB::kStageBytes;
            bool good = mbar_wait(&full[s], (it / kStages) & 1, kWaitNs);
            tc_fence_after_sync();
            if (tid == 0 && good) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kin = ks & 3;
                    mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(st + SmemB::kStageA1 + kb * 16384 + kin * 32)),
                                sdesc_k_sw128(smem_u32(ST + kb * 2048 + kin * 32)), id, ks > 0);
                }
                mma_commit(mbar1);
            }
            good = good && mbar_wait(mbar1, it & 1, kWaitNs);
            tc_fence_after_sync();
            float d1[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 0), d1);
            tmem_wait_ld();
            const int tok = (warp & 1) * 32 + lane;
            if (warp < 2) {
                // U = U0 - W S  -> U^T operand (row j, token tok)
                const __nv_bfloat16* u0 = (const __nv_bfloat16*)(st + SmemB::kStageU0) + tok * kTile;
#pragma unroll
                for (int j = 0; j < kTile; ++j)
                    *(__nv_bfloat16*)(UT + sw128_off(j, tok)) = __float2bfloat16_rn(__bfloat162float(u0[j]) - d1[j]);
                fence_proxy_async_smem();
            } else if (good) {
                // O = O0 + Q' S  -> out
                const int64_t t = seq0 + (int64_t)it * kChunk + tok;
                if (t < seq1) {
                    const __nv_bfloat16* o0 = (const __nv_bfloat16*)(st + SmemB::kStageO0) + tok * kTile;
                    uint32_t p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        p[e] = pack_bf16x2(__bfloat162float(o0[2 * e]) + d1[2 * e],
                                           __bfloat162float(o0[2 * e + 1]) + d1[2 * e + 1]);
                    uint4* dst = (uint4*)(out + ((size_t)t * H + h) * kTcD + col0);
                    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                }
            }
            tc_fence_before_sync();
            if (!bar_and(128, good)) { ok = false; break; }
            tc_fence_after_sync();
            if (tid == 0) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ss(tmem + 16, sdesc_k_sw128(smem_u32(st + SmemB::kStageKE + ks * 32)),
                                sdesc_k_sw128(smem_u32(UT + ks * 32)), id, ks > 0);
                mma_commit(mbar3);
            }
            good = mbar_wait(mbar3, it & 1, kWaitNs);
            tc_fence_after_sync();
            float d3[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 16), d3);
            tmem_wait_ld();
            const float gam = ((const float*)(st + SmemB::kStageGam))[i];
#pragma unroll
            for (int j = 0; j < kTile; ++j) S[j] = fmaf(gam, S[j], d3[j]);
            write_ST();
            fence_proxy_async_smem();
            tc_fence_before_sync();
            if (!bar_and(128, good)) { ok = false; break; }
            if (tid == 0) mbar_arrive(&empty[s]);
        }
        if (!ok) {
            *(volatile int*)s_abort = 1;
            if (tid == 0) record_status(hdr, KDA_ERR_TIMEOUT);
        } else if (final_state) {
            float4* p = (float4*)(final_state + sbase);
#pragma unroll
            for (int q4 = 0; q4 < kTile / 4; ++q4)
                p[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 32);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// [T, H, 128] bf16 tensor, box = one (chunk, head) tile of 64 tokens x 128.
static bool make_map(CUtensorMap* m, const void* base, int64_t T, int H) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)kTcD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t gstr[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)H * kTcD * 2};
    cuuint32_t box[3] = {kTcD, 1, kChunk}, es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t prefill_tc_launch(const PrefillArgs& a, int64_t T, cudaStream_t stream) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(kda_tc_intra_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SmemA::kBytes)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kda_tc_inter_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SmemB::kBytes)) != cudaSuccess) return e;
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[0], stream)) != cudaSuccess) return e;
    if (a.chunks_ub > 0 && T > 0) {
        CUtensorMap mq, mk, mv, ml;
        if (!make_map(&mq, a.q, T, a.H) || !make_map(&mk, a.k, T, a.H) || !make_map(&mv, a.v, T, a.H) ||
            !make_map(&ml, a.la, T, a.H))
            return cudaErrorInvalidValue;
        kda_tc_intra_chunk<<<dim3(a.chunks_ub, a.H), 128, SmemA::kBytes, stream>>>(
            mq, mk, mv, ml, (const __nv_bfloat16*)a.beta, a.cu, (DeviceHeader*)a.hdr, a.chunk_first, a.N, a.H,
            (uint8_t*)a.recs);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[1], stream)) != cudaSuccess) return e;
    kda_tc_inter_chunk<<<dim3((unsigned)a.N * a.H, kTiles), 160, SmemB::kBytes, stream>>>(
        a.cu, (DeviceHeader*)a.hdr, a.chunk_first, a.H, (const uint8_t*)a.recs, a.s0, (__nv_bfloat16*)a.out, a.sf);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[2], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace kda

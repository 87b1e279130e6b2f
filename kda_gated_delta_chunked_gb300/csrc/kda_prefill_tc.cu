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
// Kernel (a), one CTA per (chunk, head), 256 threads, three CTAs per SM (80
// registers, ~69 KB of shared memory, 128 TMEM columns each):
//   1. One thread starts TMA copies of k, q (and log alpha) into the
//      shared-memory places the scaled operands will take (128-byte swizzle,
//      64 tokens x 64 channels a box), first thing, ahead of the set-up (a
//      single sequence needs no table lookup for the chunk's bounds); rows past
//      the sequence end are zeroed after the copy lands.  (Per-thread 16-byte
//      cp.async pieces instead were 3% slower.)  Each thread owns 4 token rows
//      x 8 key channels: a sum of log alpha over its rows and a prefix over the
//      16 row groups through shared memory give each row's running sum.  It then
//      writes every scaled operand as bf16 with 16-byte stores over the raw
//      pieces, all token-major (no transposes): K~ = K 2^g, Q~ = Q 2^g,
//      K^ = K 2^-g (g counted from the chunk start, in log2 units), and K^end
//      straight into the record.  V goes from HBM to the tensor core untouched
//      (TMA, 128-byte swizzle), brought into L2 at the start and into shared
//      memory after the solve, over the dead A^ (loading half of it at the
//      start into 8 KB more shared memory was 1% slower).
//   2. MMA-a (M=128, N=64, K=128): [K~; Q~] K^^T gives the Gram block (rows
//      0..63) and Q~ K^T (rows 64..127) in one TMEM accumulator.
//   3. With A^[i][j] = beta_j (K~ K^T)[i][j] (j < i), the rows of
//      Y^ = [T; P T] solve  Y^ (I + A^) = [Diag(beta); P Diag(beta)]  (beta
//      folded into the columns, so the solution needs no later rescaling).
//      The solve runs in 16-column blocks from the right: the coupling to the
//      already solved blocks is one small MMA (M=128, N=16) from the bf16 Y^
//      and A^ (stored row by row, read MN-major), issued as soon as the block
//      it reads is stored; the 16 x 16 diagonal block is a right-looking fp32
//      recursion (one FMA per dependent step).  (Forming the diagonal-block
//      inverses first, so that the sequential part is only the MMAs, was
//      measured 1% slower: the recursion's work moves, it does not shrink.)
//   4. MMA-b (M=128, N=128 twice, K=64): Y^ [K~], then Y^ [V], each half in
//      the same 128 TMEM columns, K~ read MN-major from the MMA-a operand; the
//      first half's epilogue forms Q' = Q~ - P T K~.  (A
//      reference point in mid-chunk, so that K~ and K^ stay within 2^+-50,
//      needed a per-channel rescaling in the epilogue and was 5% slower.)
//   5. The records kernel (b) reads are written as ready-to-copy shared-memory
//      images: [W; Q'] (K-major, 128-byte swizzle), K^end and U0 (token-major,
//      128-byte swizzle), O0 in 16-column tiles (boxes of out), Gamma.  [W; Q']
//      and U0 / O0 are staged in shared memory (in place over the dead
//      operands) and leave in 1-D bulk stores, [W; Q'] while the second half of
//      MMA-b runs.  (A coalesced 16-byte copy
//      by all threads was 4% slower, and stores straight from the accumulator
//      rows, where every lane of a store touched its own 128-byte line, 9%.)
// Chunks whose cumulative decay from the chunk start exceeds 2^100 in some
// channel cannot use this factorisation (K^ would leave the range where the
// products stay finite in fp32); for those the Gram and Q~ K^T rows are formed
// on CUDA cores with exp(g_i - g_j) (never > 1) inside the channel sums and
// stored to TMEM where MMA-a would have put them.
//
// Kernel (b), one CTA per (sequence, head, segment of chunks), 16 consumer
// warps and a producer warp: the producer streams each chunk's record into a
// two-stage shared-memory ring with 1-D bulk copies; the consumers keep the
// whole 128 x 128 state of the head in fp32 registers (one row and 32 columns
// per thread) and per chunk one thread issues
//   MMA1 (M=128, N=128, K=128): [W; Q'] S  -> U = U0 - W S (rows 0..63),
//                                             O = O0 + Q' S (rows 64..127)
//   MMA3 (M=128, N=128, K=64):  K^end^T U  -> S <- Gamma * S + K^end^T U
// with S and U fed back to the tensor core as bf16 MN-major operands.  Long
// sequences are cut into segments that run in parallel (see the segment scan
// below the kernel (a) code); the transition passes that map each segment's
// start state to its end state take the step as one product, S <- Diag(Gamma)
// S + N S + [B | 0] with N = -K^end^T W and B = K^end^T U0 formed a chunk ahead,
// and have an MMA-issuing warp of their own.
//
// Every wait on an mbarrier is bounded; on timeout the kernel records
// KDA_ERR_TIMEOUT in the device status word, drains its own copies and exits.
#include <cudaTypedefs.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_paths.h"
#include "kda_sm100.cuh"
#include "kda_tc_record.cuh"

namespace kda {

using namespace sm100;

constexpr int kTcD = 128;                // head size handled here
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxSpanLog2 = kTcMaxSpanLog2;   // fast path if max_c (-g_C) <= 100 (log2 units, from the chunk start)

size_t tc_record_bytes() { return TcRec::kBytes; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}
// 2^x with the special-function unit's instruction (relative error ~2^-22 in
// the PTX ISA); used where x is known to lie well inside [-126, 127].
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// A read-only global load kept in program order (volatile), so that it is
// issued where written even when a later branch could skip its use.
__device__ __forceinline__ uint32_t ld_nc_u16(const void* p) {
    unsigned short r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ float bf_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf_hi(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Kernel (a)
// ---------------------------------------------------------------------------
constexpr int kAThreads = 256;
// TMEM: 128 columns (three CTAs per SM).  Until the solve ends the Gram /
// Q~ K^T block sits at columns 0..63 and the coupling accumulators at 64..111;
// then MMA-b's two halves ([K~], then [V]) use columns 0..127 in turn.
constexpr uint32_t kTmCols = 128;
constexpr uint32_t kTmGram = 0;
constexpr uint32_t kTmCpl = 64;

struct SmemA {   // byte offsets from a 1024-aligned base; ~69 KB, three CTAs per SM
    static constexpr uint32_t kOpA = 0;         // [K~; Q~], K-major 128B-swizzle, 2 K-blocks x 16 KB;
                                                // MMA-a A, then MMA-b B (MN-major), then the [W; Q'] image
    static constexpr uint32_t kOpB1 = 32768;    // MMA-a B K^, K-major, 2 K-blocks x 8 KB; then:
    static constexpr uint32_t kAt = 32768;      //   A^ by 16-column blocks, MN-major 32B-swizzle, 4 x 2 KB;
                                                //   after the solve the V tile (TMA, 2 x [64 tok x 64 ch]),
                                                //   then the U0 image
    static constexpr uint32_t kV = 32768;
    static constexpr uint32_t kAt32 = 40960;    //   diagonal 16 x 16 blocks of A^, fp32 [64 rows][16], 4 KB
    static constexpr uint32_t kY = 49152;       // Y^ = [T; P T], bf16 K-major [128 x 64], 16 KB; then the O0 image
    static constexpr uint32_t kPart = 49152;    // (before Y^) per-row-group sums of log alpha, fp32 [16][128]
    static constexpr uint32_t kGS = 32768;      // (slow path, before A^) g, fp32 [64][128], 32 KB
    static constexpr uint32_t kMisc = 65536;    // beta[64], barriers, TMEM slot, flags, g_C, scalar gates[64]
    static constexpr uint32_t kBytes = kMisc + 2304 + 1024;   // misc ends at +2304; 1024 to align the base
};

// Byte offset of (row m, column n < 16) in a 16-column block of an MN-major
// operand with 32-byte swizzle: 32-byte rows, 8-row groups of 256 bytes, the
// two 16-byte halves of a row swapped on rows 4..7 of each group.
__device__ __forceinline__ uint32_t sw32_off(uint32_t m, uint32_t n) {
    return (m >> 3) * 256u + (m & 7u) * 32u + ((((n >> 3) ^ ((m & 7u) >> 2)) & 1u) << 4) + (n & 7u) * 2u;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Column block J (16 columns) of the solve Y^ (I + A^) = RHS for row `tid`
// (threads 0..127) of Y^: the right-hand side (from the Gram / Q~ K^T
// accumulator still in TMEM columns 0..63), minus the coupling to the solved
// blocks on the right, then the in-block recursion on the fp32 diagonal block;
// stored to Y^ as bf16.  Threads 128..255 only take part in the barrier.
//
// The coupling of block J' to block ks > J' is one MMA (M=128, N=16, K=16) from
// the bf16 Y^ and A^ into TMEM columns 64 + 16 J'.  They are issued as soon as
// block ks is stored: at the start of block J, the products of block J+1 with
// every block J' <= J, the one for J itself first and committed, so each block
// waits for a single MMA; the others run during its recursion and are covered
// by the next commit (one thread's MMAs complete in order).
template <int J>
__device__ __forceinline__ void inv_block(uint8_t* sm, uint32_t tmem, const float* s_beta, uint64_t* bar,
                                          int* s_flag, uint32_t& mph, bool& abort) {
    const int tid = threadIdx.x, warp = tid >> 5;
    uint8_t* yop = sm + SmemA::kY;
    if (J < 3 && tid == 0 && !abort) {
        const uint64_t ya = sdesc_k_sw128(smem_u32(yop + (J + 1) * 32));
        const uint32_t id = idesc_bf16(128, 16, 0, 1);
        mma_bf16_ss(tmem + kTmCpl + 16 * J, ya, sdesc(smem_u32(sm + SmemA::kAt + J * 2048 + (J + 1) * 512), 2048, 256, 6),
                    id, J + 1 < 3);
        mma_commit(bar);
#pragma unroll
        for (int jt = J - 1; jt >= 0; --jt)
            mma_bf16_ss(tmem + kTmCpl + 16 * jt, ya,
                        sdesc(smem_u32(sm + SmemA::kAt + jt * 2048 + (J + 1) * 512), 2048, 256, 6), id, J + 1 < 3);
    }
    if (warp < 4) {
        float z[16];
        if (warp < 2) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) z[jj] = (16 * J + jj == tid) ? s_beta[tid] : 0.f;
        } else {
            const int i = tid - 64;
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, kTmGram + 16 * J), f);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) z[jj] = (16 * J + jj <= i) ? f[jj] * s_beta[16 * J + jj] : 0.f;
        }
        if (J < 3) {
            if (!abort && !mbar_wait(bar, mph & 1, kWaitNs)) s_flag[1] = 1;
            tc_fence_after_sync();
            float dd[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, kTmCpl + 16 * J), dd);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) z[jj] -= dd[jj];
        }
        // Right-looking: once z[m] is final, remove its share A^[m][jj] from
        // every z[jj], jj < m.  The dependent chain is one FMA per step.
        const float4* arow = (const float4*)(sm + SmemA::kAt32) + 16 * J * 4;
#pragma unroll
        for (int m = 15; m >= 1; --m) {
            const float zm = z[m];
#pragma unroll
            for (int g4 = 0; 4 * g4 < m; ++g4) {
                const float4 a = arow[m * 4 + g4];
                if (4 * g4 + 0 < m) z[4 * g4 + 0] = fmaf(-zm, a.x, z[4 * g4 + 0]);
                if (4 * g4 + 1 < m) z[4 * g4 + 1] = fmaf(-zm, a.y, z[4 * g4 + 1]);
                if (4 * g4 + 2 < m) z[4 * g4 + 2] = fmaf(-zm, a.z, z[4 * g4 + 2]);
                if (4 * g4 + 3 < m) z[4 * g4 + 3] = fmaf(-zm, a.w, z[4 * g4 + 3]);
            }
        }
        uint32_t p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = pack_bf16x2(z[2 * e], z[2 * e + 1]);
        *(uint4*)(yop + sw128_off(tid, 16 * J)) = make_uint4(p[0], p[1], p[2], p[3]);
        *(uint4*)(yop + sw128_off(tid, 16 * J + 8)) = make_uint4(p[4], p[5], p[6], p[7]);
        fence_proxy_async_smem();
    }
    if (J < 3) ++mph;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    abort = s_flag[1] != 0;
}

template <bool kScalarGate>
__global__ void __launch_bounds__(kAThreads, 3)
kda_tc_intra_chunk(const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_la,
                   const __nv_bfloat16* __restrict__ q,
                   const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ log_alpha,
                   const __nv_bfloat16* __restrict__ beta, const int32_t* __restrict__ cu,
                   DeviceHeader* __restrict__ hdr, const int32_t* __restrict__ chunk_first, int N, int H,
                   int64_t T, uint8_t* __restrict__ recs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* s_beta = (float*)(sm + SmemA::kMisc);                 // [64]
    uint64_t* bars = (uint64_t*)(sm + SmemA::kMisc + 768);       // [0] V tile, [1] MMAs, [2] inputs
    uint32_t* s_tmem = (uint32_t*)(sm + SmemA::kMisc + 800);
    int* s_flag = (int*)(sm + SmemA::kMisc + 816);                // [0] slow path, [1] abort
    float* s_gtot = (float*)(sm + SmemA::kMisc + 1024);           // [128] g_C per channel
    float* s_lg = (float*)(sm + SmemA::kMisc + 2048);             // [64] scalar gates of the chunk

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y;
    int64_t t0;
    int len, status;
    if (N == 1) {
        // One sequence starts at token 0 (a cu_seqlens that does not is flagged
        // in the status word), so the chunk's bounds follow from c alone and
        // the input loads below wait for no table.
        status = hdr->status;
        t0 = (int64_t)c * kChunk;
        if (t0 >= T) return;
        len = (int)min64(kChunk, T - t0);
    } else {
        // The status word, the chunk's sequence and its bounds are loaded
        // together; the tables are always written, so reading them before the
        // status check is safe.
        status = hdr->status;
        const int total_chunks = hdr->total_chunks;
        const int n = chunk_owner(chunk_first, N, c);
        const int64_t seq_begin = cu[n], seq_end = cu[n + 1];
        const int c_first = chunk_first[n];
        if (status != KDA_OK || c >= total_chunks) return;
        t0 = seq_begin + (int64_t)(c - c_first) * kChunk;
        len = (int)min64(kChunk, seq_end - t0);
    }

    // ---- inputs: k and q are copied by TMA into [K~; Q~] and log alpha into
    // K^ (64 tokens x 64 channels a box, 128-byte swizzle), the places where
    // the scaled operands are written over them, so no register holds them
    // meanwhile; rows past the sequence are zeroed once the copy has landed.
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
        s_flag[0] = 0;
        s_flag[1] = 0;
        mbar_arrive_expect_tx(&bars[2], kScalarGate ? 32768 : 49152);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_3d(sm + SmemA::kOpA + kb * 16384, &tm_k, 64 * kb, h, (int)t0, &bars[2]);
            tma_load_3d(sm + SmemA::kOpA + kb * 16384 + 8192, &tm_q, 64 * kb, h, (int)t0, &bars[2]);
            if (!kScalarGate) tma_load_3d(sm + SmemA::kOpB1 + kb * 8192, &tm_la, 64 * kb, h, (int)t0, &bars[2]);
        }
    }
    uint32_t braw = 0, lraw = 0;
    // beta, and with the scalar gate the chunk's 64 gates, one per thread
    // (loaded once and shared: 4 scalar loads per thread were 10% slower).
    if (tid < len) {
        braw = ld_nc_u16(beta + (size_t)(t0 + tid) * H + h);
        if (kScalarGate) lraw = ld_nc_u16(log_alpha + (size_t)(t0 + tid) * H + h);
    }
    // (a single sequence checks the status word after the prefix below, before
    // its first write, so the set-up does not wait for it)
    uint8_t* rec = recs + ((size_t)c * H + h) * TcRec::kBytes;
    if (kScalarGate && tid < kChunk) s_lg[tid] = __uint_as_float(lraw << 16);
    __syncthreads();
    if (tid == 0) {                    // V is loaded after the solve; bring it into L2 now
        tma_prefetch_3d(&tm_v, 0, h, (int)t0);
        tma_prefetch_3d(&tm_v, 64, h, (int)t0);
    }
    if (tid < kChunk) s_beta[tid] = __uint_as_float(braw << 16);
    if (warp == 0) { tmem_alloc(s_tmem, kTmCols); tmem_relinquish(); }

    // ---- pass A: thread owns rows 4R..4R+3, channels 8C..8C+7: the sum of log
    // alpha (log2 units) over its rows; pass B forms the running sums again row
    // by row (they would hold 32 registers meanwhile).
    const int R = tid >> 4, C = tid & 15;
    const uint32_t kbA = (uint32_t)C >> 3, ccA = (uint32_t)(C & 7) * 8u;
    bool in_late = false;              // the input copy outlived the wait (error path)
    if (!mbar_wait(&bars[2], 0, kWaitNs)) { s_flag[1] = 1; in_late = true; }
    if (len < kChunk) {                // rows past the sequence hold the next one's tokens: zero them
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * R + i;
            if (r >= len) {
                *(uint4*)(sm + SmemA::kOpA + kbA * 16384 + sw128_off(r, ccA)) = make_uint4(0, 0, 0, 0);
                *(uint4*)(sm + SmemA::kOpA + kbA * 16384 + sw128_off(64 + r, ccA)) = make_uint4(0, 0, 0, 0);
                if (!kScalarGate)
                    *(uint4*)(sm + SmemA::kOpB1 + kbA * 8192 + sw128_off(r, ccA)) = make_uint4(0, 0, 0, 0);
            }
        }
    }
    auto la_row = [&](int i, float (&la)[8]) {
        if (kScalarGate) {
            const float l = s_lg[4 * R + i];
#pragma unroll
            for (int e = 0; e < 8; ++e) la[e] = l;
        } else {
            unpack8(*(const uint4*)(sm + SmemA::kOpB1 + kbA * 8192 + sw128_off(4 * R + i, ccA)), la);
        }
    };
    {
        float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float la[8];
            la_row(i, la);
#pragma unroll
            for (int e = 0; e < 8; ++e) s8[e] = fmaf(la[e], kLog2e, s8[e]);
        }
        float4* part = (float4*)(sm + SmemA::kPart) + (R * kTcD + 8 * C) / 4;
        part[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
        part[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
    }
    __syncthreads();
    // Exclusive prefix over the 16 row groups, one thread per channel, in place;
    // the chunk total g_C goes to s_gtot.  A chunk whose decay from its start
    // exceeds 2^kMaxSpanLog2 in some channel takes the slow path.
    if (tid < kTcD) {
        float* pc = (float*)(sm + SmemA::kPart) + tid;
        float x[16];
#pragma unroll
        for (int rg = 0; rg < 16; ++rg) x[rg] = pc[rg * kTcD];
        float acc = 0.f;
#pragma unroll
        for (int rg = 0; rg < 16; ++rg) { pc[rg * kTcD] = acc; acc += x[rg]; }
        s_gtot[tid] = acc;
        if (-acc > kMaxSpanLog2) s_flag[0] = 1;              // any writer sets 1
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // g before this thread's rows and at row 63 (g_C), for its 8 channels.
    float gbase[8], gC[8];
    {
        const float4* part = (const float4*)(sm + SmemA::kPart);
        const float4* tot = (const float4*)s_gtot;
        const float4 a = part[(R * kTcD + 8 * C) / 4], b = part[(R * kTcD + 8 * C) / 4 + 1];
        const float4 e = tot[2 * C], f = tot[2 * C + 1];
        gbase[0] = a.x; gbase[1] = a.y; gbase[2] = a.z; gbase[3] = a.w;
        gbase[4] = b.x; gbase[5] = b.y; gbase[6] = b.z; gbase[7] = b.w;
        gC[0] = e.x; gC[1] = e.y; gC[2] = e.z; gC[3] = e.w; gC[4] = f.x; gC[5] = f.y; gC[6] = f.z; gC[7] = f.w;
    }
    const uint32_t tmem = *s_tmem;
    if (status != KDA_OK) {            // uniform; nothing has been written yet
        if (warp == 0) tmem_dealloc(tmem, kTmCols);
        if (in_late) mbar_wait(&bars[2], 0, kWaitNs);
        return;
    }
    const bool slow = s_flag[0] != 0;
    // The slow path's g scratch overlaps the prefix sums just read: all reads first.
    if (slow) __syncthreads();
    if (slow && tid == 0) hdr->pad[kHdrSlowChunk] = 1;   // some chunk needs the slow path
    if (R == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ((float*)(rec + TcRec::kGam))[8 * C + e] = exp2f(gC[e]);
    }

    // ---- pass B: scaled operands for the thread's 4 rows x 8 channels.
    {
        const uint32_t kb = (uint32_t)C >> 3, cc = (uint32_t)(C & 7) * 8u;
        uint8_t* opA = sm + SmemA::kOpA + kb * 16384;
        uint8_t* opB1 = sm + SmemA::kOpB1 + kb * 8192;
        uint8_t* ke = rec + TcRec::kKE + kb * 8192;
        float gr[8];                                       // running g_r (log2 units)
#pragma unroll
        for (int e = 0; e < 8; ++e) gr[e] = gbase[e];
        if (!slow) {
            // -g_C <= 100 and g_r lies in [g_C, 0] (log alpha <= 0), so every
            // exponent below is within [-100, 100].
            float fC[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) fC[e] = ex2_fast(gC[e]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * R + i;
                {
                    float la[8];
                    la_row(i, la);                         // read before K^ is written over it
#pragma unroll
                    for (int e = 0; e < 8; ++e) gr[e] = fmaf(la[e], kLog2e, gr[e]);
                }
                float kv[8], qv[8], km[8], qm[8], kh[8], kend[8];
                const uint32_t off = sw128_off(r, cc), offq = sw128_off(64 + r, cc);
                unpack8(*(const uint4*)(opA + off), kv);
                unpack8(*(const uint4*)(opA + offq), qv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float e1 = ex2_fast(gr[e]);      // 2^g_r
                    const float e2 = ex2_fast(-gr[e]);     // 2^-g_r
                    km[e] = kv[e] * e1;
                    qm[e] = qv[e] * e1;
                    kh[e] = kv[e] * e2;
                    kend[e] = kh[e] * fC[e];               // k 2^(g_C - g_r) <= |k|
                }
                *(uint4*)(opA + off) = pack8(km);
                *(uint4*)(opA + offq) = pack8(qm);
                *(uint4*)(opB1 + off) = pack8(kh);
                *(uint4*)(ke + off) = pack8(kend);
            }
        } else {
            // The slow path's fp32 g scratch overlays log alpha: every thread
            // reads its four rows before any of it is written.
            float gl[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float la[8];
                la_row(i, la);
#pragma unroll
                for (int e = 0; e < 8; ++e) { gr[e] = fmaf(la[e], kLog2e, gr[e]); gl[i][e] = gr[e]; }
            }
            __syncthreads();
            float* gS = (float*)(sm + SmemA::kGS);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * R + i;
                float kv[8], qv[8], km[8], qm[8], kend[8];
                const uint32_t off = sw128_off(r, cc), offq = sw128_off(64 + r, cc);
                unpack8(*(const uint4*)(opA + off), kv);
                unpack8(*(const uint4*)(opA + offq), qv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float g = gl[i][e];
                    const float e3 = exp2f(g);
                    km[e] = kv[e] * e3;
                    qm[e] = qv[e] * e3;
                    kend[e] = kv[e] * exp2f(gC[e] - g);
                    gS[r * kTcD + 8 * C + e] = g;
                }
                *(uint4*)(opA + off) = pack8(km);
                *(uint4*)(opA + offq) = pack8(qm);
                *(uint4*)(ke + off) = pack8(kend);
            }
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    uint32_t mph = 0;                 // completed phases of bars[1]
    bool abort = false;
    bool v_issued = false;            // (thread 0) the V tile copy is in flight
    if (!slow) {
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = ks & 3;
                mma_bf16_ss(tmem + kTmGram, sdesc_k_sw128(smem_u32(sm + SmemA::kOpA + kb * 16384 + kin * 32)),
                            sdesc_k_sw128(smem_u32(sm + SmemA::kOpB1 + kb * 8192 + kin * 32)), id, ks > 0);
            }
            mma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], mph & 1, kWaitNs)) s_flag[1] = 1;
        ++mph;
        tc_fence_after_sync();
    } else {
        // Rows of the Gram block (lane quarters 0,1) and of Q~ K^T (2,3) on CUDA
        // cores with exp(g_i - g_j) <= 1 inside the sums, stored to TMEM.  The
        // two warps of a lane quarter split the 64 columns.
        const float* gS = (const float*)(sm + SmemA::kGS);
        const int quarter = warp & 3, half = warp >> 2;
        const int i = (quarter & 1) * 32 + lane;
        const __nv_bfloat16* left = (quarter < 2 ? k : q) + ((size_t)(t0 + i) * H + h) * kTcD;
#pragma unroll 1
        for (int j0 = 32 * half; j0 < 32 * half + 32; j0 += 16) {
            float f[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int j = j0 + jj;
                float acc = 0.f;
                if (j <= i && i < len) {
                    const __nv_bfloat16* kj = k + ((size_t)(t0 + j) * H + h) * kTcD;
#pragma unroll 1
                    for (int c2 = 0; c2 < kTcD; ++c2)
                        acc = fmaf(__bfloat162float(left[c2]) * __bfloat162float(kj[c2]),
                                   exp2f(gS[i * kTcD + c2] - gS[j * kTcD + c2]), acc);
                }
                f[jj] = acc;
            }
            tmem_st16(tmem_addr(tmem, 32 * quarter, kTmGram + j0), f);
        }
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();                  // K^ (or g) no longer needed
    tc_fence_after_sync();
    abort = s_flag[1] != 0;

    // A^[i][j] = beta_j G[i][j] (j < i) row by row into the 16-column blocks
    // (MN-major, rows m = i), and the diagonal blocks row by row into At32.
    {
        const int quarter = warp & 3, half = warp >> 2;
        if (quarter < 2) {
            const int i = quarter * 32 + lane;
            float* at32 = (float*)(sm + SmemA::kAt32);
#pragma unroll 1
            for (int j0 = 32 * half; j0 < 32 * half + 32; j0 += 16) {
                float f[16];
                tmem_ld16(tmem_addr(tmem, 32 * quarter, kTmGram + j0), f);
                tmem_wait_ld();
                float a[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) a[jj] = (j0 + jj < i) ? s_beta[j0 + jj] * f[jj] : 0.f;
                if ((j0 >> 4) == (i >> 4)) {           // diagonal block: row i, fp32
                    float4* dst = (float4*)(at32 + i * 16);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4)
                        dst[e4] = make_float4(a[4 * e4], a[4 * e4 + 1], a[4 * e4 + 2], a[4 * e4 + 3]);
                }
                uint8_t* blk = sm + SmemA::kAt + (j0 >> 4) * 2048;
                float lo[8], hi[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) { lo[e] = a[e]; hi[e] = a[8 + e]; }
                *(uint4*)(blk + sw32_off(i, 0)) = pack8(lo);
                *(uint4*)(blk + sw32_off(i, 8)) = pack8(hi);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // ---- Y^ (I + A^) = [Diag(beta); P Diag(beta)], 16-column blocks from the right.
    inv_block<3>(sm, tmem, s_beta, &bars[1], s_flag, mph, abort);
    inv_block<2>(sm, tmem, s_beta, &bars[1], s_flag, mph, abort);
    inv_block<1>(sm, tmem, s_beta, &bars[1], s_flag, mph, abort);
    inv_block<0>(sm, tmem, s_beta, &bars[1], s_flag, mph, abort);

    // ---- MMA-b, first half: Y^ [K~] -> [W; P T K~] in columns 0..127 (the Gram
    // and coupling accumulators are dead).  V is loaded into the dead A^ region.
    if (tid == 0 && !abort) {
        mbar_arrive_expect_tx(&bars[0], 16384);
        tma_load_3d(sm + SmemA::kV, &tm_v, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + SmemA::kV + 8192, &tm_v, 64, h, (int)t0, &bars[0]);
        v_issued = true;
        const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(sm + SmemA::kY + ks * 32)),
                        sdesc(smem_u32(sm + SmemA::kOpA + ks * 2048), 16384, 1024, 2), id, ks > 0);
        mma_commit(&bars[1]);
    }
    if (!abort && !mbar_wait(&bars[1], mph & 1, kWaitNs)) s_flag[1] = 1;
    ++mph;
    tc_fence_after_sync();
    __syncthreads();
    abort = s_flag[1] != 0;

    // ---- epilogue, first half.  Lane quarters 0,1: rows 0..63 = W; quarters
    // 2,3: rows 64..127 = P T K~ -> Q' = Q~ - P T K~.  The two warps of a quarter
    // split the columns; the [W; Q'] image is staged in place over [K~; Q~].
    const int quarter = warp & 3, half = warp >> 2;
    const int i = (quarter & 1) * 32 + lane;      // token row within the chunk
    const bool top = quarter < 2;
    if (!abort) {
        uint8_t* a1 = sm + SmemA::kOpA;
        const uint8_t* qm = sm + SmemA::kOpA;
#pragma unroll 1
        for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * quarter, c0), f);
            tmem_wait_ld();
            const uint32_t kb = c0 >> 6, kin = c0 & 63;
            const int row = top ? i : 64 + i;
            if (!top) {                                // Q' = Q~ - P T K~
                float q0[8], q1[8];
                unpack8(*(const uint4*)(qm + kb * 16384 + sw128_off(row, kin)), q0);
                unpack8(*(const uint4*)(qm + kb * 16384 + sw128_off(row, kin + 8)), q1);
#pragma unroll
                for (int e = 0; e < 8; ++e) { f[e] = q0[e] - f[e]; f[8 + e] = q1[e] - f[8 + e]; }
            }
            float lo[8], hi[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) { lo[e] = f[e]; hi[e] = f[8 + e]; }
            *(uint4*)(a1 + kb * 16384 + sw128_off(row, kin)) = pack8(lo);
            *(uint4*)(a1 + kb * 16384 + sw128_off(row, kin + 8)) = pack8(hi);
        }
    }
    fence_proxy_async_smem();          // the [W; Q'] image is visible to the bulk copy engine
    tc_fence_before_sync();
    __syncthreads();                   // the first half's accumulator has been read
    tc_fence_after_sync();

    // ---- MMA-b, second half: Y^ [V] -> [U0; O0] in columns 0..127; the issuing
    // thread waits for the V tile first.
    if (tid == 0 && !abort && !mbar_wait(&bars[0], 0, kWaitNs)) { s_flag[1] = 1; abort = true; }
    if (tid == 0 && !abort) {
        const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(sm + SmemA::kY + ks * 32)),
                        sdesc(smem_u32(sm + SmemA::kV + ks * 2048), 8192, 1024, 2), id, ks > 0);
        mma_commit(&bars[1]);
        bulk_s2g(rec + TcRec::kA1, sm + SmemA::kOpA, 32768);
        bulk_commit();
    }
    __syncthreads();
    abort = s_flag[1] != 0;
    if (!abort && !mbar_wait(&bars[1], mph & 1, kWaitNs)) s_flag[1] = 1;
    ++mph;
    tc_fence_after_sync();
    __syncthreads();
    abort = s_flag[1] != 0;

    // ---- epilogue, second half: the U0 image (rows 0..63; token-major, two
    // 64-channel blocks in 128-byte swizzle, an MN-major operand of the chain)
    // and the O0 image (rows 64..127; 16-column tiles) over the dead V tile and Y^.
    if (!abort) {
        uint8_t* uo = sm + SmemA::kAt + (top ? 0 : TcRec::kO0 - TcRec::kU0);   // U0 | O0 images
#pragma unroll 1
        for (int t = 4 * half; t < 4 * half + 4; ++t) {
            float f[16];
            tmem_ld16(tmem_addr(tmem, 32 * quarter, t * kTile), f);
            tmem_wait_ld();
            float lo[8], hi[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) { lo[e] = f[e]; hi[e] = f[8 + e]; }
            if (top) {
                const uint32_t c = (uint32_t)t * kTile;
                uint8_t* ub = uo + (c >> 6) * 8192u;
                *(uint4*)(ub + sw128_off(i, c & 63u)) = pack8(lo);
                *(uint4*)(ub + sw128_off(i, (c & 63u) + 8u)) = pack8(hi);
            } else {
                uint4* dst = (uint4*)(uo + t * TcRec::kTileBytes + i * (kTile * 2));
                dst[0] = pack8(lo);
                dst[1] = pack8(hi);
            }
        }
    } else if (tid == 0) {
        record_status(hdr, KDA_ERR_TIMEOUT);
    }
    fence_proxy_async_smem();          // the staged images are visible to the bulk copy engine
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmCols);
    if (tid == 0) {
        if (!abort) {                  // the [W; Q'] and [U0; O0] images go to the record in two bulk stores
            static_assert(SmemA::kAt + 2 * (TcRec::kO0 - TcRec::kU0) <= SmemA::kMisc, "staging fits");
            static_assert(TcRec::kU0 - TcRec::kA1 >= 32768 && TcRec::kO0 + 16384 <= TcRec::kGam, "record spans");
            bulk_s2g(rec + TcRec::kU0, sm + SmemA::kAt, 32768);
            bulk_commit();
        }
        bulk_wait_read_all();          // shared memory stays valid until the engine has read it
        if (v_issued) mbar_wait(&bars[0], 0, kWaitNs);   // the V tile copy has landed before exit
        if (in_late) mbar_wait(&bars[2], 0, kWaitNs);
    }
}

// ---------------------------------------------------------------------------
// Kernel (b): the chain over chunks, one CTA per (sequence, head, segment)
// ---------------------------------------------------------------------------
// Segments split one sequence's chunks so that long sequences occupy every SM.
// Segment 0 is [0, L0) and segment p >= 1 is [L0 + (p-1) L, L0 + p L):
//   launch 1: segment 0 runs the output pass (OUT, N = 128) from the initial
//      state, writing its outputs and its end state S_start(1); at the same
//      time every segment p = 1 .. segs-2 runs the transition pass (N = 256)
//      from the augmented state X = [0 | I]: it ends at [B_p | M_p], the
//      affine map  S_end = M_p S_start + B_p  of the segment;
//   launch 2 (phase B): S_start(p+1) = M_p S_start(p) + B_p, sequential over
//      p >= 1, fp32;
//   launch 3: segments 1 .. segs-1 run the output pass from their start
//      states; the last writes the final state.
// Segment 0 is longer (L0 ~ 1.2 L) because its output pass shares launch 1
// with the transitions, whose steps take longer (measured: 1.0 and 1.3 were
// 2% and 3% slower on the chain).  A sequence that gets one
// segment is the plain chain (launch 1 only).  Planning uses a fixed SM count
// so that the workspace size depends on (N, H, T) only.
constexpr int kPlanSMs = 152;
constexpr int kChainWarps = 16;                 // consumer warps (4 per TMEM lane quarter)
constexpr int kChainThreads = 32 * kChainWarps + 32;   // consumers and the record producer
constexpr int kOLeader = 64;                    // lane 0 of warp 2: issues the output pass's TMA stores

struct ScanPlan {
    int len0;         // chunks of segment 0
    int len;          // chunks of every later segment
    int segs_max;     // segments of the longest possible sequence
};
// Shortest segment, in chunks.  Segments are as long as the SM count allows
// (1,929 / 1,607 chunks on a 2^20-token sequence of 16 heads); the floor only
// matters for short sequences, whose walk is a few steps per segment.
constexpr int64_t kMinSegChunks = 8;

static ScanPlan scan_plan(int N, int H, int64_t T) {
    ScanPlan p;
    const int64_t chunks_max = (T + kChunk - 1) / kChunk;
    const int64_t nh = (int64_t)N * H;
    const int64_t target = nh > 0 ? kPlanSMs / nh : 1;    // CTAs per (sequence, head) in launches 1 and 3
    if (target < 2 || chunks_max <= 2 * kMinSegChunks) {
        p.len0 = (int)(chunks_max > 0 ? chunks_max : 1);
        p.len = 1;
        p.segs_max = 1;
        return p;
    }
    int64_t len = (10 * chunks_max + 10 * target + 11) / (10 * target + 12);   // chunks_max / (target + 1.2)
    if (len < kMinSegChunks) len = kMinSegChunks;  // below this the launches and the scan cost more than they save
    int64_t len0 = (12 * len + 9) / 10;
    if (len0 + target * len < chunks_max) len0 = chunks_max - target * len;
    if (len0 > chunks_max) len0 = chunks_max;
    p.len0 = (int)len0;
    p.len = (int)len;
    p.segs_max = chunks_max <= len0 ? 1 : 1 + (int)((chunks_max - len0 + len - 1) / len);
    return p;
}
// Segment scratch per (sequence, head, segment): M_p fp32 [128][128] (contiguous,
// so that the scan moves it with one bulk copy), B_p fp32 [128][128], and
// S_start fp32 [128][128].
constexpr size_t kSegM = 0, kSegB = (size_t)kTcD * kTcD * 4, kSegMB = 2 * kSegB;
constexpr size_t kSegS = (size_t)kTcD * kTcD * 4, kSegBytes = kSegMB + kSegS;

// Number of segments of a sequence of nch chunks, and the first chunk of segment p.
__host__ __device__ __forceinline__ int seg_count(int nch, int len0, int len) {
    return nch <= len0 ? 1 : 1 + (nch - len0 + len - 1) / len;
}
__host__ __device__ __forceinline__ int seg_begin(int p, int len0, int len) {
    return p == 0 ? 0 : len0 + (p - 1) * len;
}

size_t tc_extra_bytes(int N, int H, int64_t T) {
    const ScanPlan p = scan_plan(N, H, T);
    return p.segs_max > 1 ? (size_t)N * H * p.segs_max * kSegBytes : 0;
}

// Output pass: a two-stage ring of whole records, the X and U operands.
struct SmemO {   // byte offsets from a 1024-aligned base
    static constexpr uint32_t kA1 = 0, kKE = 32768, kU0 = 49152, kO0 = 65536, kGam = 81920;
    static constexpr uint32_t kTx = kGam + 512;                      // bytes copied per stage
    static constexpr uint32_t kStageBytes = (kTx + 1023) / 1024 * 1024;
    static constexpr uint32_t kX = 2 * kStageBytes;                  // X operand, MN-major, [128 x 128]
    static constexpr uint32_t kU = kX + 128 * 128 * 2;               // U operand, MN-major, [64 x 128]
    static constexpr uint32_t kMisc = kU + 64 * 128 * 2;
    static constexpr uint32_t kBytes = kMisc + 256 + 1024;
};

// Byte offset of (row, col) in an MN-major 128-byte-swizzle operand whose
// 64-column atoms hold `rows` rows each.
__device__ __forceinline__ uint32_t mn_off(uint32_t row, uint32_t col, uint32_t rows) {
    return (col >> 6) * rows * 128u + sw128_off(row, col & 63u);
}

// Arguments shared by the chain launches.
struct ChainArgs {
    CUtensorMap tm_out;          // out [T, H, 128] bf16, box 16 columns x 1 head x 64 tokens
    int has_tm_out;
    const int32_t* cu;
    DeviceHeader* hdr;
    const int32_t* chunk_first;
    int H, len0, len, segs_max;
    const uint8_t* recs;
    const float* initial_state;
    __nv_bfloat16* out;
    float* final_state;
    uint8_t* segbuf;
    const int32_t* snap_slot;
    float* snaps;
};

// One CTA's output pass over segment p of sequence-head blockIdx.x, from the
// segment's start state: the outputs of its chunks and its end state.
__device__ __forceinline__ void out_segment(const ChainArgs& A, int p) {
    const int32_t* __restrict__ cu = A.cu;
    DeviceHeader* __restrict__ hdr = A.hdr;
    const int32_t* __restrict__ chunk_first = A.chunk_first;
    const int H = A.H, segs_max = A.segs_max;
    const uint8_t* __restrict__ recs = A.recs;
    const float* __restrict__ initial_state = A.initial_state;
    __nv_bfloat16* __restrict__ out = A.out;
    float* __restrict__ final_state = A.final_state;
    uint8_t* __restrict__ segbuf = A.segbuf;
    const int32_t* __restrict__ snap_slot = A.snap_slot;
    float* __restrict__ snaps = A.snaps;
    using L = SmemO;
    constexpr int NX = 128;                            // state columns
    constexpr int kCols = NX / 4;                      // columns per consumer warp
    constexpr int kLdB = 2;                            // TMEM loads in flight per wait
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(sm + L::kMisc);     // [2]
    uint64_t* empty = full + 2;                      // [2]
    uint64_t* mbar = empty + 2;
    uint32_t* s_tmem = (uint32_t*)(mbar + 1);
    int* s_abort = (int*)(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (hdr->status != KDA_OK) return;
    const int nh = blockIdx.x, n = nh / H, h = nh % H;
    const int c_seq = chunk_first[n], nch = chunk_first[n + 1] - c_seq;
    const int segs = seg_count(nch, A.len0, A.len);
    if (p >= segs) return;
    const int cb = seg_begin(p, A.len0, A.len);                 // chunk range within the sequence
    const int ce = min(nch, seg_begin(p + 1, A.len0, A.len));
    const int nsteps = ce - cb;
    const int64_t seq0 = cu[n], seq1 = cu[n + 1];
    uint8_t* seg = segbuf ? segbuf + ((size_t)nh * segs_max + p) * kSegBytes : nullptr;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(mbar, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) { tmem_alloc(s_tmem, 2 * NX); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;

    if (warp == kChainWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nsteps; ++it) {
                const int s = it & 1;
                if (it >= 2 && !mbar_wait(&empty[s], ((it >> 1) - 1) & 1, kWaitNs)) {
                    *(volatile int*)s_abort = 1;
                    break;
                }
                if (*(volatile int*)s_abort) break;
                const uint8_t* rec = recs + ((size_t)(c_seq + cb + it) * H + h) * TcRec::kBytes;
                uint8_t* st = sm + s * L::kStageBytes;
                mbar_arrive_expect_tx(&full[s], L::kTx);
                bulk_g2s(st + L::kA1, rec + TcRec::kA1, 32768, &full[s]);
                bulk_g2s(st + L::kKE, rec + TcRec::kKE, 16384, &full[s]);
                bulk_g2s(st + L::kU0, rec + TcRec::kU0, 16384, &full[s]);
                bulk_g2s(st + L::kO0, rec + TcRec::kO0, 16384, &full[s]);
                bulk_g2s(st + L::kGam, rec + TcRec::kGam, 512, &full[s]);
                issued = it + 1;
            }
            for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
                mbar_wait(&full[it & 1], (it >> 1) & 1, kWaitNs);
        }
    } else if (warp < kChainWarps) {
        // ---------------- consumers: rows 32q..32q+31, columns [col0, col0 + kCols) ----------------
        const int q = warp & 3, g = warp >> 2;
        const int i = 32 * q + lane;                 // key channel (row of S / X)
        const int tok = (q & 1) * 32 + lane;          // token row of the U / O halves
        const int col0 = g * kCols;
        float X[kCols];
        {
            const float* src = (p == 0) ? initial_state + ((size_t)nh * kTcD + i) * kTcD
                                        : (const float*)(seg + kSegMB) + (size_t)i * kTcD;
            if (p == 0 && !initial_state) {
#pragma unroll
                for (int j = 0; j < kCols; ++j) X[j] = 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < kCols; j += 4) {
                    const float4 v = *(const float4*)(src + col0 + j);
                    X[j] = v.x; X[j + 1] = v.y; X[j + 2] = v.z; X[j + 3] = v.w;
                }
            }
        }
        uint8_t* XO = sm + L::kX;
        uint8_t* UO = sm + L::kU;
        auto write_X = [&](float gam) {
#pragma unroll
            for (int j = 0; j < kCols; j += 8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = gam * X[j + e];
                *(uint4*)(XO + mn_off(i, col0 + j, 128)) = pack8(v);
            }
        };
        const uint32_t id1 = idesc_bf16(128, NX, 0, 1);     // [W; Q'] K-major, X MN-major
        const uint32_t id3 = idesc_bf16(128, NX, 1, 1);     // K^end MN-major, U MN-major
        uint32_t ph = 0;
        write_X(1.f);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        bool ok = bar_and(32 * kChainWarps, true);
        for (int it = 0; it < nsteps && ok; ++it) {
            const int s = it & 1;
            const uint8_t* st = sm + s * L::kStageBytes;
            // snapshot request for the state after this chunk
            const int snap_m = snap_slot ? snap_slot[c_seq + cb + it] : -1;
            bool good = mbar_wait(&full[s], (it >> 1) & 1, kWaitNs);
            tc_fence_after_sync();
            if (tid == 0 && good) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kin = ks & 3;
                    mma_bf16_ss(tmem, sdesc_k_sw128(smem_u32(st + L::kA1 + kb * 16384 + kin * 32)),
                                sdesc(smem_u32(XO + ks * 2048), 16384, 1024, 2), id1, ks > 0);
                }
                mma_commit(mbar);
            }
            // This thread's U0 (U warps) or O0 (O warps) pieces are read while
            // MMA1 runs (the stage has landed).
            uint4 pre[4];
            {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t c = (uint32_t)(col0 + 16 * hh);
                    if (q < 2) {           // U0: two 64-channel blocks, 128-byte swizzle
                        const uint8_t* ub = st + L::kU0 + (c >> 6) * 8192u;
                        pre[2 * hh] = *(const uint4*)(ub + sw128_off(tok, c & 63u));
                        pre[2 * hh + 1] = *(const uint4*)(ub + sw128_off(tok, (c & 63u) + 8u));
                    } else {               // O0: 16-column tiles
                        const uint8_t* p = st + L::kO0 + tok * (kTile * 2) + (c >> 4) * TcRec::kTileBytes;
                        pre[2 * hh] = *(const uint4*)p;
                        pre[2 * hh + 1] = *(const uint4*)(p + 16);
                    }
                }
            }
            good = good && mbar_wait(mbar, ph & 1, kWaitNs);
            ++ph;
            tc_fence_after_sync();
            if (q < 2) {
                // U = U0 - W X
#pragma unroll
                for (int j2 = 0; j2 < kCols; j2 += 16 * kLdB) {
                  float dd[kLdB][16];
#pragma unroll
                  for (int hh = 0; hh < kLdB; ++hh) tmem_ld16(tmem_addr(tmem, 32 * q, col0 + j2 + 16 * hh), dd[hh]);
                  tmem_wait_ld();
#pragma unroll
                  for (int hh = 0; hh < kLdB; ++hh) {
                    const float (&d)[16] = dd[hh];
                    const int c = col0 + j2 + 16 * hh;
                    float lo[8], hi[8], a[8], b[8];
                    unpack8(pre[2 * (j2 / 16 + hh)], a);
                    unpack8(pre[2 * (j2 / 16 + hh) + 1], b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) { lo[e] = a[e] - d[e]; hi[e] = b[e] - d[8 + e]; }
                    *(uint4*)(UO + mn_off(tok, c, 64)) = pack8(lo);
                    *(uint4*)(UO + mn_off(tok, c + 8, 64)) = pack8(hi);
                  }
                }
                fence_proxy_async_smem();
            } else {
                // O = O0 + Q' S -> out.  The TMEM loads are warp-collective: every
                // lane takes part, only the stores of real tokens are predicated.
                // A full chunk's O goes back into the stage's O0 tiles (same layout
                // as a [64 x 16] box of out) and leaves with TMA stores; a partial
                // last chunk is stored row by row.
                const int64_t t = seq0 + (int64_t)(cb + it) * kChunk + tok;
                const bool full = A.has_tm_out && seq0 + (int64_t)(cb + it + 1) * kChunk <= seq1;
                const bool store = good && t < seq1;
#pragma unroll
                for (int j2 = 0; j2 < kCols; j2 += 16 * kLdB) {
                  float dd[kLdB][16];
#pragma unroll
                  for (int hh = 0; hh < kLdB; ++hh) tmem_ld16(tmem_addr(tmem, 32 * q, col0 + j2 + 16 * hh), dd[hh]);
                  tmem_wait_ld();
#pragma unroll
                  for (int hh = 0; hh < kLdB; ++hh) {
                    const float (&d)[16] = dd[hh];
                    const int c = col0 + j2 + 16 * hh;
                    float a[8], b[8];
                    unpack8(pre[2 * (j2 / 16 + hh)], a);
                    unpack8(pre[2 * (j2 / 16 + hh) + 1], b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) { a[e] += d[e]; b[e] += d[8 + e]; }
                    if (full) {
                        uint4* dst = (uint4*)(st + L::kO0 + (c >> 4) * TcRec::kTileBytes + tok * (kTile * 2));
                        dst[0] = pack8(a);
                        dst[1] = pack8(b);
                    } else if (store) {
                        uint4* dst = (uint4*)(out + ((size_t)t * H + h) * kTcD + c);
                        dst[0] = pack8(a);
                        dst[1] = pack8(b);
                    }
                  }
                }
                if (full) fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            // MMA3 needs U only: the U warps meet on their own barrier and it is
            // issued while the O warps finish the outputs (and one of them issues
            // their TMA stores); everyone meets at the step's end.
            if (q < 2) {
                good = bar_and_id(2, 32 * kChainWarps / 2, good);
            } else {
                good = bar_and_id(3, 32 * kChainWarps / 2, good);
                if (tid == kOLeader && good && A.has_tm_out && seq0 + (int64_t)(cb + it + 1) * kChunk <= seq1) {
#pragma unroll
                    for (int tl = 0; tl < kTcD / kTile; ++tl)
                        tma_store_3d(&A.tm_out, st + L::kO0 + tl * TcRec::kTileBytes, tl * kTile, h,
                                     (int)(seq0 + (int64_t)(cb + it) * kChunk));
                    bulk_commit();
                }
            }
            tc_fence_after_sync();
            if (tid == 0 && good) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ss(tmem + NX, sdesc(smem_u32(st + L::kKE + ks * 2048), 8192, 1024, 2),
                                sdesc(smem_u32(UO + ks * 2048), 8192, 1024, 2), id3, ks > 0);
                mma_commit(mbar);
            }
            good = good && mbar_wait(mbar, ph & 1, kWaitNs);
            ++ph;
            tc_fence_after_sync();
            const float gam = ((const float*)(st + L::kGam))[i];
#pragma unroll
            for (int j = 0; j < kCols; j += 16 * kLdB) {
                float d[kLdB][16];
#pragma unroll
                for (int hh = 0; hh < kLdB; ++hh) tmem_ld16(tmem_addr(tmem, 32 * q, NX + col0 + j + 16 * hh), d[hh]);
                tmem_wait_ld();
#pragma unroll
                for (int hh = 0; hh < kLdB; ++hh)
#pragma unroll
                    for (int e = 0; e < 16; ++e) X[j + 16 * hh + e] = fmaf(gam, X[j + 16 * hh + e], d[hh][e]);
            }
            if (snap_m >= 0 && good) {
                float* dst = snaps + (((size_t)snap_m * H + h) * kTcD + i) * kTcD + col0;
#pragma unroll
                for (int j = 0; j < kCols; j += 4) *(float4*)(dst + j) = make_float4(X[j], X[j + 1], X[j + 2], X[j + 3]);
            }
            write_X(1.f);
            fence_proxy_async_smem();
            if (tid == kOLeader) bulk_wait_read_all();   // the stage's O tiles have been stored
            tc_fence_before_sync();
            ok = bar_and(32 * kChainWarps, good);
            if (ok && tid == 0) mbar_arrive(&empty[s]);
        }
        if (!ok) {
            *(volatile int*)s_abort = 1;
            if (tid == 0) record_status(hdr, KDA_ERR_TIMEOUT);
        } else {
            float* dst = nullptr;
            if (p == segs - 1) {
                if (final_state) dst = final_state + ((size_t)nh * kTcD + i) * kTcD + col0;
            } else if (p == 0) {       // segment 0 hands its end state to segment 1
                dst = (float*)(segbuf + ((size_t)nh * segs_max + 1) * kSegBytes + kSegMB) + (size_t)i * kTcD + col0;
            }
            if (dst) {
#pragma unroll
                for (int j = 0; j < kCols; j += 4) *(float4*)(dst + j) = make_float4(X[j], X[j + 1], X[j + 2], X[j + 3]);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * NX);
}

// Transition pass of segment p (1 .. segs-2) on X = [0 | I] (128 x 256), which
// ends as [B_p | M_p].  One chunk's step X <- Diag(Gamma) X + K^end^T (U0' - W X),
// with U0' = [U0 | 0], is written as
//   X <- Diag(Gamma) X + N X + [B | 0],   N = -K^end^T W,  B = K^end^T U0,
// so that only the product N X depends on X.  -K^end^T [W | U0] = [N | -B] of
// chunk c+1 (one MMA group, N = 256, A negated, into TMEM columns 256..511)
// runs on the tensor core right behind N_c X; the consumers then turn its
// first half into the bf16 K-major operand N over the dead W / U0 of that
// chunk's stage and fold Diag(Gamma) and -B into the register state, which is
// carried as Y = -X (Y <- Diag(Gamma) Y + N Y - B; X = -Y at the end).
// A step is one MMA group (M = 128, N = 256, K = 128) and one pass over the
// state.  A warp of its own issues the MMAs, so that no consumer warp waits on
// the tensor core's queue, and the consumer warps hand each step's operands
// to it through an mbarrier rather than a CTA-wide barrier.
struct SmemT {   // byte offsets from a 1024-aligned base
    static constexpr uint32_t kW = 0;            // W, then U0: the B operand [W | U0], MN-major,
    static constexpr uint32_t kU0 = 16384;       //   4 atoms of [64 tok x 64 ch] at 8 KB (record layouts)
    static constexpr uint32_t kKE = 32768;       // K^end (record layout): A operand, MN-major
    static constexpr uint32_t kN = 0;            // then N = -K^end^T W over W / U0: K-major, 2 x [128 x 64]
    static constexpr uint32_t kGam = 49152;      // Gamma, 128 fp32
    static constexpr uint32_t kTx = kGam + 512;  // bytes copied per stage
    static constexpr uint32_t kStageBytes = (kTx + 1023) / 1024 * 1024;
    static constexpr int kStages = 3;
    static constexpr uint32_t kX = kStages * kStageBytes;    // X, MN-major [128 x 256] bf16
    static constexpr uint32_t kMisc = kX + 128 * 256 * 2;
    static constexpr uint32_t kBytes = kMisc + 128 + 1024;
};
constexpr uint32_t kTmD = 0, kTmE = 256, kTmEB = 384;     // TMEM columns: N X; N = -K^end^T W; -B = -K^end^T U0
constexpr int kIssuerWarp = kChainWarps + 1;              // the transition's MMA issuer
constexpr int kChainFirstThreads = 32 * kChainWarps + 64;  // consumers, producer, issuer

__device__ __forceinline__ void trans_segment(const ChainArgs& A, int p) {
    using L = SmemT;
    DeviceHeader* __restrict__ hdr = A.hdr;
    const int32_t* __restrict__ chunk_first = A.chunk_first;
    const int H = A.H;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(sm + L::kMisc);     // [kStages]
    uint64_t* empty = full + L::kStages;             // [kStages]
    uint64_t* mE = empty + L::kStages;               // K^end^T [W | U0] of a chunk
    uint64_t* mD = mE + 1;                           // N X of a chunk
    uint64_t* mC = mD + 1;                           // the consumer warps: a step's operands are in place
    uint32_t* s_tmem = (uint32_t*)(mC + 1);
    int* s_abort = (int*)(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (hdr->status != KDA_OK) return;
    const int nh = blockIdx.x, n = nh / H, h = nh % H;
    const int c_seq = chunk_first[n], nch = chunk_first[n + 1] - c_seq;
    const int segs = seg_count(nch, A.len0, A.len);
    if (p == 0 || p >= segs - 1) return;
    const int cb = seg_begin(p, A.len0, A.len);
    const int nsteps = min(nch, seg_begin(p + 1, A.len0, A.len)) - cb;   // >= 1: an inner segment
    uint8_t* seg = A.segbuf + ((size_t)nh * A.segs_max + p) * kSegBytes;

    if (tid == 0) {
        for (int s = 0; s < L::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(mE, 1);
        mbar_init(mD, 1);
        mbar_init(mC, kChainWarps);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) { tmem_alloc(s_tmem, 512); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    uint8_t* XO = sm + L::kX;

    if (warp == kChainWarps) {
        // ---------------- producer: W (rows 0..63 of [W; Q']), U0, K^end, Gamma ----------------
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nsteps; ++it) {
                const int s = it % L::kStages, use = it / L::kStages;
                if (use >= 1 && !mbar_wait(&empty[s], (use - 1) & 1, kWaitNs)) {
                    *(volatile int*)s_abort = 1;
                    break;
                }
                if (*(volatile int*)s_abort) break;
                const uint8_t* rec = A.recs + ((size_t)(c_seq + cb + it) * H + h) * TcRec::kBytes;
                uint8_t* st = sm + s * L::kStageBytes;
                mbar_arrive_expect_tx(&full[s], L::kTx);
                bulk_g2s(st + L::kW, rec + TcRec::kA1, 8192, &full[s]);
                bulk_g2s(st + L::kW + 8192, rec + TcRec::kA1 + 16384, 8192, &full[s]);
                bulk_g2s(st + L::kU0, rec + TcRec::kU0, 16384, &full[s]);
                bulk_g2s(st + L::kKE, rec + TcRec::kKE, 16384, &full[s]);
                bulk_g2s(st + L::kGam, rec + TcRec::kGam, 512, &full[s]);
                issued = it + 1;
            }
            for (int it = issued - L::kStages < 0 ? 0 : issued - L::kStages; it < issued; ++it)
                mbar_wait(&full[it % L::kStages], (it / L::kStages) & 1, kWaitNs);
        }
    } else if (warp == kIssuerWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            auto issue_E = [&](int it) -> bool {
                const uint8_t* st = sm + (it % L::kStages) * L::kStageBytes;
                if (!mbar_wait(&full[it % L::kStages], (it / L::kStages) & 1, kWaitNs)) return false;
                tc_fence_after_sync();
                const uint32_t id = idesc_bf16(128, 256, 1, 1) | (1u << 13);   // A negated: [N | -B]
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ss(tmem + kTmE, sdesc(smem_u32(st + L::kKE + ks * 2048), 8192, 1024, 2),
                                sdesc(smem_u32(st + L::kW + ks * 2048), 8192, 1024, 2), id, ks > 0);
                mma_commit(mE);
                return true;
            };
            bool good = issue_E(0);
            for (int it = 0; it < nsteps && good; ++it) {
                // the consumers have written N_it and X_it and read the accumulators
                if (!mbar_wait(mC, it & 1, kWaitNs) || *(volatile int*)s_abort) { good = false; break; }
                tc_fence_after_sync();
                const uint8_t* st = sm + (it % L::kStages) * L::kStageBytes;
                const uint32_t id = idesc_bf16(128, 256, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kin = ks & 3;
                    mma_bf16_ss(tmem + kTmD, sdesc_k_sw128(smem_u32(st + L::kN + kb * 16384 + kin * 32)),
                                sdesc(smem_u32(XO + ks * 2048), 16384, 1024, 2), id, ks > 0);
                }
                mma_commit(mD);
                if (it + 1 < nsteps && !issue_E(it + 1)) good = false;
            }
            if (!good) *(volatile int*)s_abort = 1;
        }
    } else {
        // ---------------- consumers: row i of the state, columns [col0, col0 + 64) ----------------
        // (X[] holds Y = -X; the MMA operand written from it is Y as well)
        const int q = warp & 3, g = warp >> 2;
        const int i = 32 * q + lane;
        const int col0 = g * 64;
        float X[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) X[j] = (col0 + j == kTcD + i) ? -1.f : 0.f;   // Y = -[0 | I]
        auto write_X = [&]() {
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = X[j + e];
                *(uint4*)(XO + mn_off(i, col0 + j, 128)) = pack8(v);
            }
        };
        // Once chunk it's K^end^T [W | U0] has landed: N (negated, bf16) over
        // its stage's dead W / U0, and X <- Diag(Gamma) X + [B | 0] in registers.
        auto prepare = [&](int it, bool good) -> bool {
            good = good && mbar_wait(mE, it & 1, kWaitNs);
            tc_fence_after_sync();
            uint8_t* st = sm + (it % L::kStages) * L::kStageBytes;
            {
                float f0[16], f1[16];
                tmem_ld16(tmem_addr(tmem, 32 * q, kTmE + 32 * g), f0);
                tmem_ld16(tmem_addr(tmem, 32 * q, kTmE + 32 * g + 16), f1);
                tmem_wait_ld();
                uint8_t* nb = st + L::kN + (uint32_t)(g >> 1) * 16384u;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = m < 2 ? f0[8 * m + e] : f1[8 * (m - 2) + e];
                    *(uint4*)(nb + sw128_off(i, (uint32_t)(32 * (g & 1) + 8 * m))) = pack8(v);
                }
            }
            const float gam = ((const float*)(st + L::kGam))[i];
            if (col0 < kTcD) {           // Y <- Diag(Gamma) Y + (-B)
#pragma unroll
                for (int j = 0; j < 64; j += 32) {
                    float b0[16], b1[16];
                    tmem_ld16(tmem_addr(tmem, 32 * q, kTmEB + col0 + j), b0);
                    tmem_ld16(tmem_addr(tmem, 32 * q, kTmEB + col0 + j + 16), b1);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        X[j + e] = fmaf(gam, X[j + e], b0[e]);
                        X[j + 16 + e] = fmaf(gam, X[j + 16 + e], b1[e]);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) X[j] *= gam;
            }
            return good;
        };
        // This warp's share of a step's operands is in place and its accumulator
        // reads are done: one arrival per warp.
        auto hand_off = [&](bool good) {
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (!good) *(volatile int*)s_abort = 1;
                mbar_arrive(mC);
            }
        };

        bool good = true;
        write_X();
        good = __all_sync(0xffffffffu, prepare(0, good));
        hand_off(good);
        for (int it = 0; it < nsteps && good; ++it) {
            good = !*(volatile int*)s_abort && mbar_wait(mD, it & 1, kWaitNs);
            good = __all_sync(0xffffffffu, good);
            if (!good) break;
            tc_fence_after_sync();
            if (tid == 0) mbar_arrive(&empty[it % L::kStages]);   // N_it X_it has read its stage
#pragma unroll
            for (int j = 0; j < 64; j += 32) {
                float d0[16], d1[16];
                tmem_ld16(tmem_addr(tmem, 32 * q, kTmD + col0 + j), d0);
                tmem_ld16(tmem_addr(tmem, 32 * q, kTmD + col0 + j + 16), d1);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) { X[j + e] += d0[e]; X[j + 16 + e] += d1[e]; }
            }
            write_X();
            if (it + 1 < nsteps) {
                good = __all_sync(0xffffffffu, prepare(it + 1, good));
                hand_off(good);
            }
        }
        if (!good) {
            *(volatile int*)s_abort = 1;
            if (lane == 0) record_status(hdr, KDA_ERR_TIMEOUT);
        } else {
            // X = -Y: columns 0..127 are B_p, 128..255 are M_p
            float* dst = (float*)(seg + (col0 >= kTcD ? kSegM : kSegB)) + (size_t)i * kTcD + (col0 & (kTcD - 1));
#pragma unroll
            for (int j = 0; j < 64; j += 4) *(float4*)(dst + j) = make_float4(-X[j], -X[j + 1], -X[j + 2], -X[j + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (*(volatile int*)s_abort && tid == 0) record_status(hdr, KDA_ERR_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Launch 1: segment 0's output pass (blockIdx.y == 0) beside the transition
// passes of segments 1 .. segs-2 (blockIdx.y = p).
__global__ void __launch_bounds__(kChainFirstThreads, 1) kda_tc_chain_first(const __grid_constant__ ChainArgs A) {
    if (A.hdr->status != KDA_OK) return;
    if (blockIdx.y == 0) out_segment(A, 0);
    else trans_segment(A, blockIdx.y);
}

constexpr uint32_t kChainFirstSmem = SmemO::kBytes > SmemT::kBytes ? SmemO::kBytes : SmemT::kBytes;

// Launch 3: the output passes of segments 1 .. segs-1 (p = blockIdx.y + 1).
__global__ void __launch_bounds__(kChainThreads, 1) kda_tc_chain_rest(const __grid_constant__ ChainArgs A) {
    if (A.hdr->status != KDA_OK) return;
    out_segment(A, blockIdx.y + 1);
}

// Phase B: S_start(p+1) = M_p S_start(p) + B_p for p = 1 .. segs-2, from
// S_start(1) (segment 0's end state), for one (sequence, head) and a
// 16-column block of the state (columns of S are independent), fp32.  Each
// M_p (64 KB) comes into shared memory with one bulk copy, two segments ahead
// of its use; thread (r0, c) forms rows r0, r0 + 16, ... of column c.
constexpr int kScanThreads = 256;
constexpr uint32_t kScanSmem = 2 * 65536 + kTcD * 16 * 4 + 64 + 1024;
__global__ void __launch_bounds__(kScanThreads, 1)
kda_tc_scan_states(const int32_t* __restrict__ chunk_first, DeviceHeader* __restrict__ hdr, int H, int len0,
                   int len, uint8_t* __restrict__ segbuf, int segs_max) {
    if (hdr->status != KDA_OK) return;
    const int nh = blockIdx.x, n = nh / H, cblk = blockIdx.y * 16;
    const int nch = chunk_first[n + 1] - chunk_first[n];
    const int segs = seg_count(nch, len0, len);
    if (segs < 3) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* Mbuf = (float*)sm;                               // [2][128][128]
    float* S = (float*)(sm + 2 * 65536);                    // [128][16]
    uint64_t* bar = (uint64_t*)(sm + 2 * 65536 + kTcD * 16 * 4);
    const int tid = threadIdx.x, c = tid & 15, r0 = tid >> 4;
    auto seg = [&](int p) { return segbuf + ((size_t)nh * segs_max + p) * kSegBytes; };
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int p = 1; p <= 2 && p + 1 < segs; ++p) {
            mbar_arrive_expect_tx(&bar[p - 1], 65536);
            bulk_g2s(Mbuf + (p - 1) * kTcD * kTcD, seg(p) + kSegM, 65536, &bar[p - 1]);
        }
    }
    const float* S1 = (const float*)(seg(1) + kSegMB);
    for (int e = tid; e < kTcD * 16; e += kScanThreads) {
        const int r = e >> 4, cc = e & 15;
        S[e] = S1[(size_t)r * kTcD + cblk + cc];
    }
    __syncthreads();
    bool good = true;
    int p = 1;
    for (; p + 1 < segs; ++p) {
        const int b = (p - 1) & 1;
        const float* Bp = (const float*)(seg(p) + kSegB);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = Bp[(size_t)(r0 + 16 * j) * kTcD + cblk + c];
        good = bar_and(kScanThreads, mbar_wait(&bar[b], ((p - 1) >> 1) & 1, kWaitNs));   // uniform
        if (!good) break;
        const float* M = Mbuf + b * kTcD * kTcD;
        for (int k = 0; k < kTcD; k += 4) {
            const float s0 = S[k * 16 + c], s1 = S[(k + 1) * 16 + c], s2 = S[(k + 2) * 16 + c],
                        s3 = S[(k + 3) * 16 + c];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 m = *(const float4*)(M + (r0 + 16 * j) * kTcD + k);
                acc[j] = fmaf(m.x, s0, fmaf(m.y, s1, fmaf(m.z, s2, fmaf(m.w, s3, acc[j]))));
            }
        }
        __syncthreads();                                     // S and this M buffer fully read
        if (tid == 0 && p + 3 <= segs - 1) {                 // M_{p+2} into the buffer just read
            mbar_arrive_expect_tx(&bar[b], 65536);
            bulk_g2s(Mbuf + b * kTcD * kTcD, seg(p + 2) + kSegM, 65536, &bar[b]);
        }
        float* Snext = (float*)(seg(p + 1) + kSegMB);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = r0 + 16 * j;
            S[r * 16 + c] = acc[j];
            Snext[(size_t)r * kTcD + cblk + c] = acc[j];
        }
        __syncthreads();
    }
    if (!good && tid == 0) {
        record_status(hdr, KDA_ERR_TIMEOUT);
        // the copies still in flight land before exit
        for (int q = p; q <= p + 1 && q + 1 < segs; ++q) mbar_wait(&bar[(q - 1) & 1], ((q - 1) >> 1) & 1, kWaitNs);
    }
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

// k, q, log alpha, V [T, H, 128] bf16; box = 64 tokens x 64 channels of one
// head, 128-byte swizzle (the K-major operand layout of the first intra-chunk
// product for k and q, the MN-major one of the second for V).
// out [T, H, 128] bf16; box = 16 channels x 1 head x 64 tokens, no swizzle
// (the layout of a U0 / O0 record tile).
static bool make_out_map(CUtensorMap* m, void* base, int64_t T, int H) {
    auto enc = encode_fn();
    if (!enc || T <= 0) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)kTcD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t gstr[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)H * kTcD * 2};
    cuuint32_t box[3] = {kTile, 1, kChunk}, es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_v_map(CUtensorMap* m, const void* base, int64_t T, int H) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)kTcD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t gstr[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)H * kTcD * 2};
    cuuint32_t box[3] = {64, 1, kChunk}, es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_make_tile_map(CUtensorMap* m, const void* base, int64_t T, int H) { return make_v_map(m, base, T, H); }

cudaError_t prefill_tc_launch(const PrefillArgs& a, int64_t T, cudaStream_t stream) {
    cudaError_t e;
    auto intra = a.la_scalar ? kda_tc_intra_chunk<true> : kda_tc_intra_chunk<false>;
    if ((e = cudaFuncSetAttribute(intra, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SmemA::kBytes)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kda_tc_chain_first, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kChainFirstSmem)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kda_tc_chain_rest, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SmemO::kBytes)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kda_tc_scan_states, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kScanSmem)) != cudaSuccess) return e;
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[0], stream)) != cudaSuccess) return e;
    if (a.chunks_ub > 0 && T > 0) {
        CUtensorMap mv;
        if (!make_v_map(&mv, a.v, T, a.H)) return cudaErrorInvalidValue;
        CUtensorMap mk, mq, ml;
        if (!make_v_map(&mk, a.k, T, a.H) || !make_v_map(&mq, a.q, T, a.H)) return cudaErrorInvalidValue;
        if (a.la_scalar) ml = mk;
        else if (!make_v_map(&ml, a.la, T, a.H)) return cudaErrorInvalidValue;
        intra<<<dim3(a.chunks_ub, a.H), kAThreads, SmemA::kBytes, stream>>>(
            mv,
            mk, mq, ml,
            (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.la,
            (const __nv_bfloat16*)a.beta, a.cu, (DeviceHeader*)a.hdr, a.chunk_first, a.N, a.H, T, (uint8_t*)a.recs);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[1], stream)) != cudaSuccess) return e;
    const ScanPlan plan = scan_plan(a.N, a.H, T);
    ChainArgs ca;
    memset(&ca, 0, sizeof(ca));
    ca.has_tm_out = make_out_map(&ca.tm_out, a.out, T, a.H) ? 1 : 0;
    ca.cu = a.cu; ca.hdr = (DeviceHeader*)a.hdr; ca.chunk_first = a.chunk_first; ca.H = a.H;
    ca.len0 = plan.len0; ca.len = plan.len; ca.segs_max = plan.segs_max;
    ca.recs = (const uint8_t*)a.recs; ca.initial_state = a.s0; ca.out = (__nv_bfloat16*)a.out;
    ca.final_state = a.sf; ca.segbuf = plan.segs_max > 1 ? (uint8_t*)a.extra : nullptr;
    ca.snap_slot = a.snap_slot; ca.snaps = a.snaps;
    const unsigned nh = (unsigned)a.N * a.H;
    const unsigned ylaunch = plan.segs_max > 1 ? (unsigned)plan.segs_max - 1 : 1;
    kda_tc_chain_first<<<dim3(nh, ylaunch), kChainFirstThreads, kChainFirstSmem, stream>>>(ca);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (plan.segs_max > 1) {
        if (plan.segs_max > 2) {
            kda_tc_scan_states<<<dim3(nh, kTcD / 16), kScanThreads, kScanSmem, stream>>>(
                a.chunk_first, (DeviceHeader*)a.hdr, a.H, plan.len0, plan.len, ca.segbuf, plan.segs_max);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        kda_tc_chain_rest<<<dim3(nh, ylaunch), kChainThreads, SmemO::kBytes, stream>>>(ca);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[2], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace kda

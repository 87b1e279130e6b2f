// kda_backward_tc.cu -- reverse mode of the KDA prefill on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA), bf16 inputs, head size 128.
//
// The pages give no backward ("Kimi Delta Attention" deep dive, section 06:
// the chunked form serves training and prefill).  This is the chain rule taken
// through the chunk algebra of the forward (section 06 matrix products inside
// a chunk, the state of section 03 carried between chunks).  For a chunk with
// start state S, end-state gradient dS' and output gradient dO:
//
//   across chunks, last to first:
//     dS = Diag(Gamma) dS' + Q~^T dO - W^T dU,   dU = K^end dS' + P^T dO
//        = Diag(Gamma) dS' - W^T (K^end dS') + Q'^T dO        (Q' = Q~ - P W)
//   inside a chunk (M = (I + A)^-1, T = M Diag(beta)):
//     dU  = K^end dS' + P^T dO            dK^end = U dS'^T
//     dP  = LowerIncl(dO U^T)             dQ~ = dO S^T + dP K^
//     dW  = -dU S^T                       dT  = dW K~^T + dU V^T
//     dV  = T^T dU                        dA  = StrictLower(-M^T (dT T^T))
//     dbeta = colsum(M o dT) + rowsum(StrictLower(G) o dA),   dG = Diag(beta) dA
//     dK~ = T^T dW + dG K^                dK^ = dP^T Q~ + dG^T K~
//   and through the decays (g the running sum of log alpha, g_C its chunk total):
//     dk = dK~ e^g + dK^ e^-g + dK^end e^(g_C - g),   dq = dQ~ e^g
//     dg = dK~ o K~ - dK^ o K^ + dQ~ o Q~ - dK^end o K^end
//     dlog alpha_i = sum_{r >= i} dg_r + colsum(dK^end o K^end) + dGamma o Gamma,
//     dGamma = rowsum(dS' o S).
//
// Three launches (after the tensor-core forward has run with every chunk's end
// state saved, see backward_tc_launch):
//   kda_tc_bwd_chain   one CTA per (sequence, head) walks its chunks in reverse:
//                      per chunk MMA-r1 (K^end dS') and MMA-r2
//                      ([W; Q']^T [-K^end dS'; dO]) on tcgen05, the gradient
//                      dS held in fp32 registers, and writes dS' of every chunk.
//   kda_tc_bwd_chunk   one CTA per (chunk, head) recomputes the chunk's
//                      operands, solves M = (I + A)^-1 in fp32 and forms every
//                      gradient above with twelve tcgen05 products; the small
//                      64 x 64 products behind dA run on CUDA cores in fp32.
// Chunks whose decay from the chunk start exceeds 2^100 in some channel cannot
// use the factorised products; the forward flags them in the workspace header
// and both kernels then return at once, leaving the call to the CUDA-core
// backward (launched after them with the same flag).
//
// Every wait on an mbarrier is bounded; on timeout a kernel records
// KDA_ERR_TIMEOUT in the device status word and returns.
#include <string.h>

#include "kda_common.cuh"
#include "kda_paths.h"
#include "kda_sm100.cuh"
#include "kda_tc_record.cuh"

namespace kda {

using namespace sm100;

namespace {

constexpr int kD = 128;
constexpr uint64_t kWait = 2000000000ull;        // 2 s per wait
constexpr float kL2e = 1.4426950408889634f;

// Byte offset of (row r, column c) in a bf16 tile stored as 64-column atoms
// of `rows` rows x 128 bytes with the 128-byte swizzle.  Such a tile serves as
// a K-major A (M = rows) or B (N = rows) operand and, read the other way, as an
// MN-major one.
__device__ __forceinline__ uint32_t toff(uint32_t r, uint32_t c, uint32_t rows) {
    return (c >> 6) * rows * 128u + sw128_off(r, c & 63u);
}
__device__ __forceinline__ uint32_t pk2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint4 pk8(const float* f) {
    return make_uint4(pk2(f[0], f[1]), pk2(f[2], f[3]), pk2(f[4], f[5]), pk2(f[6], f[7]));
}
// 2^x with the special-function unit's instruction; every argument here lies in
// [-100, 100] (the chunks these kernels take have decays within 2^100).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bflo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bfhi(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }
__device__ __forceinline__ void unpk8(const uint4& v, float* f) {
    f[0] = bflo(v.x); f[1] = bfhi(v.x); f[2] = bflo(v.y); f[3] = bfhi(v.y);
    f[4] = bflo(v.z); f[5] = bfhi(v.z); f[6] = bflo(v.w); f[7] = bfhi(v.w);
}
// K-major operand descriptor of K-step ks (16 elements) of a tile with
// `rows`-row atoms; MN-major descriptor of K-step ks of a tile whose 64-wide
// MN atoms are `pitch` bytes apart.
__device__ __forceinline__ uint64_t dk_(const uint8_t* base, int ks, uint32_t rows) {
    return sdesc_k_sw128(smem_u32(base + (ks >> 2) * rows * 128u + (ks & 3) * 32u));
}
__device__ __forceinline__ uint64_t dmn(const uint8_t* base, int ks, uint32_t pitch) {
    return sdesc(smem_u32(base + ks * 2048u), pitch, 1024, 2);
}

}  // namespace

// ---------------------------------------------------------------------------
// Reverse chain: one CTA per (sequence, head)
// ---------------------------------------------------------------------------
struct RcSmem {
    static constexpr uint32_t kA1 = 0;          // [W; Q'] record image (32 KB)
    static constexpr uint32_t kKE = 32768;      // K^end record image (16 KB)
    static constexpr uint32_t kDO = 49152;      // dO tile, 2 x [64 tok x 64 ch] (TMA)
    static constexpr uint32_t kGam = 65536;     // Gamma (512 B)
    static constexpr uint32_t kStage = 66560;   // per stage, 1024-aligned
    static constexpr uint32_t kX = 2 * kStage;  // dS' as bf16, MN-major [128 x 128], two buffers
    static constexpr uint32_t kNDV = kX + 65536;   // -K^end dS', MN-major [64 x 128]
    static constexpr uint32_t kMisc = kNDV + 16384;
    static constexpr uint32_t kBytes = kMisc + 256 + 1024;
    static constexpr uint32_t kTx = 32768 + 16384 + 16384 + 512;
};
constexpr int kRcWarps = 16;                    // consumer warps (4 per TMEM lane quarter)
constexpr int kRcThreads = 32 * kRcWarps + 32;

struct RcArgs {
    CUtensorMap tm_do;           // d_out [T, H, 128] bf16, 64 x 64 boxes, 128-byte swizzle
    const int32_t* cu;
    DeviceHeader* hdr;
    const int32_t* chunk_first;
    int H;
    const uint8_t* recs;         // the forward's records
    const float* dfinal;         // dLoss / dfinal_state or null
    uint8_t* dsend;              // [chunks, H] gradient of each chunk's end state, bf16 operand tiles
                                 //   (128 x 128, two 64-column atoms of 128 rows, 128-byte swizzle)
    float* ds0;                  // dLoss / dinitial_state or null
};

__global__ void __launch_bounds__(kRcThreads, 1) kda_tc_bwd_chain(const __grid_constant__ RcArgs A) {
    DeviceHeader* __restrict__ hdr = A.hdr;
    if (hdr->status != KDA_OK || hdr->pad[kHdrSlowChunk] != 0) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(sm + RcSmem::kMisc);
    uint64_t* empty = full + 2;
    uint64_t* mbar = empty + 2;
    uint32_t* s_tmem = (uint32_t*)(mbar + 1);
    int* s_abort = (int*)(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = A.H, nh = blockIdx.x, n = nh / H, h = nh % H;
    const int c_seq = A.chunk_first[n], nch = A.chunk_first[n + 1] - c_seq;
    const int64_t seq0 = A.cu[n];

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(mbar, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) { tmem_alloc(s_tmem, 256); tmem_relinquish(); }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;

    if (warp == kRcWarps) {
        // ---------------- producer: records and dO tiles, last chunk first ----------------
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nch; ++it) {
                const int s = it & 1;
                if (it >= 2 && !mbar_wait(&empty[s], ((it >> 1) - 1) & 1, kWait)) {
                    *(volatile int*)s_abort = 1;
                    break;
                }
                if (*(volatile int*)s_abort) break;
                const int cl = nch - 1 - it;
                const uint8_t* rec = A.recs + ((size_t)(c_seq + cl) * H + h) * TcRec::kBytes;
                uint8_t* st = sm + s * RcSmem::kStage;
                mbar_arrive_expect_tx(&full[s], RcSmem::kTx);
                bulk_g2s(st + RcSmem::kA1, rec + TcRec::kA1, 32768, &full[s]);
                bulk_g2s(st + RcSmem::kKE, rec + TcRec::kKE, 16384, &full[s]);
                bulk_g2s(st + RcSmem::kGam, rec + TcRec::kGam, 512, &full[s]);
                const int tok = (int)(seq0 + (int64_t)cl * kChunk);
                tma_load_3d(st + RcSmem::kDO, &A.tm_do, 0, h, tok, &full[s]);
                tma_load_3d(st + RcSmem::kDO + 8192, &A.tm_do, 64, h, tok, &full[s]);
                issued = it + 1;
            }
            for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
                mbar_wait(&full[it & 1], (it >> 1) & 1, kWait);
        }
    } else {
        // ---------------- consumers: row i of dS (a key channel), 32 columns ----------------
        const int q = warp & 3, g = warp >> 2;
        const int i = 32 * q + lane;
        const int tok = (q & 1) * 32 + lane;
        const int col0 = 32 * g;
        float X[32];
        if (A.dfinal) {
            const float* src = A.dfinal + ((size_t)nh * kD + i) * kD + col0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v = *(const float4*)(src + j);
                X[j] = v.x; X[j + 1] = v.y; X[j + 2] = v.z; X[j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) X[j] = 0.f;
        }
        uint8_t* NDV = sm + RcSmem::kNDV;
        auto write_X = [&](int b) {
            uint8_t* XO = sm + RcSmem::kX + b * 32768;
#pragma unroll
            for (int j = 0; j < 32; j += 8) *(uint4*)(XO + toff(i, col0 + j, 128)) = pk8(&X[j]);
        };
        const uint32_t id1 = idesc_bf16(128, 128, 0, 1);
        const uint32_t id2 = idesc_bf16(128, 128, 1, 1);
        uint32_t ph = 0;
        write_X(0);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        bool ok = bar_and(32 * kRcWarps, true);
        for (int it = 0; it < nch && ok; ++it) {
            const int s = it & 1;
            const int c = c_seq + nch - 1 - it;
            const uint8_t* st = sm + s * RcSmem::kStage;
            uint8_t* XO = sm + RcSmem::kX + (it & 1) * 32768;     // dS' of this chunk, bf16
            if (tid == 0) {
                // the gradient of this chunk's end state, for the per-chunk kernel: the
                // operand tile itself, stored by the bulk-copy engine while MMA-r1 reads it
                bulk_s2g(A.dsend + ((size_t)c * H + h) * 32768, XO, 32768);
                bulk_commit();
            }
            bool good = mbar_wait(&full[s], (it >> 1) & 1, kWait);
            tc_fence_after_sync();
            if (tid == 0 && good) {
                // MMA-r1: rows 0..63 = K^end dS' (rows 64..127 read past K^end: unused)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ss(tmem, dk_(st + RcSmem::kKE, ks, 64), dmn(XO, ks, 16384), id1, ks > 0);
                mma_commit(mbar);
            }
            good = good && mbar_wait(mbar, ph & 1, kWait);
            ++ph;
            tc_fence_after_sync();
            if (q < 2) {
#pragma unroll
                for (int j2 = 0; j2 < 32; j2 += 16) {
                    float d[16];
                    tmem_ld16(tmem_addr(tmem, 32 * q, col0 + j2), d);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) d[e] = -d[e];
                    *(uint4*)(NDV + toff(tok, col0 + j2, 64)) = pk8(&d[0]);
                    *(uint4*)(NDV + toff(tok, col0 + j2 + 8, 64)) = pk8(&d[8]);
                }
                fence_proxy_async_smem();
            }
            // the other dS' buffer is written below: its store (two chunks back) has read it
            if (tid == 0) bulk_wait_read_1();
            tc_fence_before_sync();
            good = bar_and(32 * kRcWarps, good);
            tc_fence_after_sync();
            if (tid == 0 && good) {
                // MMA-r2: [W; Q']^T [-K^end dS'; dO]  (K = 64 W rows, then 64 Q' rows)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t b = ks < 4 ? dmn(NDV, ks, 8192) : dmn(st + RcSmem::kDO, ks - 4, 8192);
                    mma_bf16_ss(tmem + 128, dmn(st + RcSmem::kA1, ks, 16384), b, id2, ks > 0);
                }
                mma_commit(mbar);
            }
            good = good && mbar_wait(mbar, ph & 1, kWait);
            ++ph;
            tc_fence_after_sync();
            const float gam = ((const float*)(st + RcSmem::kGam))[i];
#pragma unroll
            for (int j = 0; j < 32; j += 16) {
                float d[16];
                tmem_ld16(tmem_addr(tmem, 32 * q, 128 + col0 + j), d);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) X[j + e] = fmaf(gam, X[j + e], d[e]);
            }
            write_X((it + 1) & 1);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            ok = bar_and(32 * kRcWarps, good);
            if (ok && tid == 0) mbar_arrive(&empty[s]);
        }
        if (tid == 0) bulk_wait_all();
        if (!ok) {
            *(volatile int*)s_abort = 1;
            if (tid == 0) record_status(hdr, KDA_ERR_TIMEOUT);
        } else if (A.ds0) {
            float* dst = A.ds0 + ((size_t)nh * kD + i) * kD + col0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *(float4*)(dst + j) = make_float4(X[j], X[j + 1], X[j + 2], X[j + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// Per-chunk gradients: one CTA per (chunk, head), 256 threads, 1 CTA per SM
// ---------------------------------------------------------------------------
// Shared memory, byte offsets from a 1024-aligned base.  bf16 operand tiles
// (64-column atoms, 128-byte swizzle), then the regions they are reused for.
struct PcSmem {
    static constexpr uint32_t kKQ = 0;          // [K~; Q~] 128 x 128 (atoms of 128 rows)
    static constexpr uint32_t kDD = 32768;      // [dO; dU] 128 x 128 (dO by TMA into rows 0..63)
    static constexpr uint32_t kSS = 65536;      // S 128 x 128; later dW (64 x 128), dP, dG (64 x 64 each);
                                                //   at the end dg fp32 [64][128].  (Phase 0: prefix sums.)
    static constexpr uint32_t kDS = 98304;      // M fp32 [64][64] (solve), then dS' 128 x 128; later
                                                //   dT / dA fp32 [64][68], M fp32 [64][68], M^T fp32 [64][64],
                                                //   X1 fp32 [64][64]; at the end g fp32 [64][128], dK~ fp32 [64][132]
    static constexpr uint32_t kVT = 131072;     // V 64 x 128 (TMA)
    static constexpr uint32_t kKE = 147456;     // K^end 64 x 128
    static constexpr uint32_t kWU = 163840;     // A-bar fp32 [64][64] (solve), then -W, then U, 64 x 128
    static constexpr uint32_t kZ0 = 180224;     // zeros 64 x 64 (the first M atom of [0; T^T])
    static constexpr uint32_t kTT = 188416;     // T 64 x 64
    static constexpr uint32_t kPT = 196608;     // P 64 x 64; later prefix sums, column partials
    static constexpr uint32_t kKH = 204800;     // K^ 64 x 128
    static constexpr uint32_t kMisc = 221184;   // six fp32 vectors (2 KB), then barriers and the TMEM slot
    static constexpr uint32_t kBytes = kMisc + 2048 + 64 + 1024;
    // late reuse
    static constexpr uint32_t kDW = kSS, kDP = kSS + 16384, kDG = kSS + 24576;
    static constexpr uint32_t kDT = kDS, kMM = kDS + 17408, kMT = kDS + 34816, kX1 = kDS + 51200;
    static constexpr uint32_t kG = kDS, kDKT = kDS + 32768;
};
static_assert(PcSmem::kX1 + 16384 <= PcSmem::kZ0, "late fp32 scratch stays clear of the zero tile");
static_assert(PcSmem::kDKT + 64 * 132 * 4 <= PcSmem::kZ0, "dK~ exchange stays clear of the zero tile");
static_assert(PcSmem::kBytes <= 227 * 1024, "shared memory");
constexpr int kPcThreads = 256;
constexpr int kLd = 68;                       // padded row of the fp32 64 x 64 matrices

template <bool kScalarGate>
__global__ void __launch_bounds__(kPcThreads, 1)
kda_tc_bwd_chunk(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                 const __nv_bfloat16* __restrict__ log_alpha, const __nv_bfloat16* __restrict__ beta,
                 const int32_t* __restrict__ cu, DeviceHeader* __restrict__ hdr,
                 const int32_t* __restrict__ chunk_first, int N, int H, const float* __restrict__ s0,
                 const float* __restrict__ snaps, const uint8_t* __restrict__ dsend, float* __restrict__ dq,
                 float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ dla,
                 float* __restrict__ dbeta) {
    using L = PcSmem;
    if (hdr->status != KDA_OK || hdr->pad[kHdrSlowChunk] != 0) return;
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= hdr->total_chunks) return;
    const int n = chunk_owner(chunk_first, N, c);
    const int c_first = chunk_first[n];
    const int64_t t0 = (int64_t)cu[n] + (int64_t)(c - c_first) * kChunk;
    const int len = (int)min64(kChunk, (int64_t)cu[n + 1] - t0);
    const float* S_src = c > c_first ? snaps + ((size_t)(c - 1) * H + h) * kD * kD
                                     : (s0 ? s0 + ((size_t)n * H + h) * kD * kD : nullptr);
    const uint8_t* dS_src = dsend + ((size_t)c * H + h) * 32768;   // bf16 operand tile of dS'

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* s_beta = (float*)(sm + L::kMisc);            // [64]
    float* s_gC = s_beta + 64;                          // [128] g_C, log2 units
    float* s_dgam = s_gC + 128;                         // [128] dGamma
    float* s_dbeta = s_dgam + 128;                      // [64]
    float* s_lg = s_dbeta + 64;                         // [64] scalar gates
    float* s_cs = s_lg + 64;                            // [64] colsum(M o dT)
    uint64_t* bars = (uint64_t*)(sm + L::kMisc + 2048); // [0] TMA, [1] MMA
    uint32_t* s_tmem = (uint32_t*)(bars + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, hcol = warp >> 2;

    // ---- phase 0: loads, running sums of log alpha, scaled operands ----
    const int R = tid >> 4, C = tid & 15;
    const size_t rs = (size_t)H * kD;
    const size_t base = ((size_t)t0 * H + h) * kD + 8 * C;
    uint4 kr[4], qr[4], lr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * R + i;
        kr[i] = qr[i] = lr[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < len) {
            kr[i] = *(const uint4*)(k + base + (size_t)r * rs);
            qr[i] = *(const uint4*)(q + base + (size_t)r * rs);
            if (!kScalarGate) lr[i] = *(const uint4*)(log_alpha + base + (size_t)r * rs);
        }
    }
    if (tid < kChunk) {
        const bool in = tid < len;
        s_beta[tid] = in ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
        if (kScalarGate) s_lg[tid] = in ? __bfloat162float(log_alpha[(size_t)(t0 + tid) * H + h]) : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    {   // zero tile
        uint4* z = (uint4*)(sm + L::kZ0);
        z[tid] = make_uint4(0u, 0u, 0u, 0u);
        z[tid + 256] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 32768 + 32768);
        tma_load_3d(sm + L::kVT, &tm_v, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + L::kVT + 8192, &tm_v, 64, h, (int)t0, &bars[0]);
        tma_load_3d(sm + L::kDD, &tm_do, 0, h, (int)t0, &bars[0]);
        tma_load_3d(sm + L::kDD + 16384, &tm_do, 64, h, (int)t0, &bars[0]);
        bulk_g2s(sm + L::kDS, dS_src, 32768, &bars[0]);
        if (S_src) bulk_prefetch_l2(S_src, kD * kD * 4);
    }
    if (warp == 0) { tmem_alloc(s_tmem, 512); tmem_relinquish(); }

    // running sum of log alpha (log2 units) within the thread's 4 rows, then an
    // exclusive prefix over the 16 row groups (the forward's own scheme)
    float gl[4][8];
    {
        float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float la[8];
            if (kScalarGate) {
                const float l = s_lg[4 * R + i];
#pragma unroll
                for (int e = 0; e < 8; ++e) la[e] = l;
            } else {
                unpk8(lr[i], la);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) { s8[e] = fmaf(la[e], kL2e, s8[e]); gl[i][e] = s8[e]; }
        }
        float4* part = (float4*)(sm + L::kSS) + (R * kD + 8 * C) / 4;
        part[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
        part[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
    }
    __syncthreads();
    if (tid < kD) {
        float* pc = (float*)(sm + L::kSS) + tid;
        float x[16];
#pragma unroll
        for (int rg = 0; rg < 16; ++rg) x[rg] = pc[rg * kD];
        float acc = 0.f;
#pragma unroll
        for (int rg = 0; rg < 16; ++rg) { pc[rg * kD] = acc; acc += x[rg]; }
        s_gC[tid] = acc;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const uint32_t R0 = tmem, R1 = tmem + 128, R2 = tmem + 256, R3 = tmem + 384;
    {
        const float* part = (const float*)(sm + L::kSS) + R * kD + 8 * C;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * R + i;
            float kv[8], qv[8], kt[8], qt[8], kh[8], ke[8];
            unpk8(kr[i], kv);
            unpk8(qr[i], qv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float g = part[e] + gl[i][e];
                const float e1 = ex2(g), e2 = ex2(-g);
                kt[e] = kv[e] * e1;
                qt[e] = qv[e] * e1;
                kh[e] = kv[e] * e2;
                ke[e] = kv[e] * ex2(s_gC[8 * C + e] - g);
            }
            *(uint4*)(sm + L::kKQ + toff(r, 8 * C, 128)) = pk8(kt);
            *(uint4*)(sm + L::kKQ + toff(64 + r, 8 * C, 128)) = pk8(qt);
            *(uint4*)(sm + L::kKH + toff(r, 8 * C, 64)) = pk8(kh);
            *(uint4*)(sm + L::kKE + toff(r, 8 * C, 64)) = pk8(ke);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    uint32_t mph = 0;
    bool tma_done = false;
    // All threads wait for the MMAs committed so far; the result is uniform.
    auto mma_done = [&](bool ok) -> bool {
        bool gd = ok && mbar_wait(&bars[1], mph & 1, kWait);
        ++mph;
        tc_fence_after_sync();
        gd = bar_and(kPcThreads, gd);
        return gd;
    };
    auto cta_sync = [&]() {
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
    };
    bool ok = true;

    // ---- phase 1: [K~; Q~] K^^T -> Gram G (rows 0..63) and Q~ K^^T (rows 64..127) ----
    if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R0, dk_(sm + L::kKQ, ks, 128), dk_(sm + L::kKH, ks, 64), idesc_bf16(128, 64), ks > 0);
        mma_commit(&bars[1]);
    }
    ok = mma_done(ok);
    if (ok) {
        // A-bar[i][j] = beta_i G[i][j] (j < i), fp32; P = LowerIncl(Q~ K^^T) as bf16
#pragma unroll
        for (int j0 = 32 * hcol; j0 < 32 * hcol + 32; j0 += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R0, 32 * quarter, j0), f);
            tmem_wait_ld();
            if (quarter < 2) {
                const int i = 32 * quarter + lane;
                const float bi = s_beta[i];
                float* dst = (float*)(sm + L::kWU) + i * 64 + j0;
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    float4 v;
                    v.x = (j0 + 4 * e4 + 0 < i) ? bi * f[4 * e4 + 0] : 0.f;
                    v.y = (j0 + 4 * e4 + 1 < i) ? bi * f[4 * e4 + 1] : 0.f;
                    v.z = (j0 + 4 * e4 + 2 < i) ? bi * f[4 * e4 + 2] : 0.f;
                    v.w = (j0 + 4 * e4 + 3 < i) ? bi * f[4 * e4 + 3] : 0.f;
                    *(float4*)(dst + 4 * e4) = v;
                }
            } else {
                const int i = 32 * (quarter - 2) + lane;
                float p[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) p[e] = (j0 + e <= i) ? f[e] : 0.f;
                *(uint4*)(sm + L::kPT + toff(i, j0, 64)) = pk8(&p[0]);
                *(uint4*)(sm + L::kPT + toff(i, j0 + 8, 64)) = pk8(&p[8]);
            }
        }
        fence_proxy_async_smem();
    }
    cta_sync();

    // ---- phase 2: M = (I + A-bar)^-1 in fp32, by 16 x 16 blocks: the four
    //      diagonal blocks D_i = (I + A-bar_ii)^-1 by a right-looking recursion
    //      (one row per thread, warps 0, 1), then the blocks below the
    //      diagonal, distance d = 1, 2, 3 in turn, from (I + A-bar) M = I:
    //        M_ij = -D_i sum_{k=j}^{i-1} A-bar_ik M_kj   (all threads). ----
    {
        const float* Ab = (const float*)(sm + L::kWU);          // A-bar, [64][64]
        float* Mw = (float*)(sm + L::kSS);                      // M, [64][64] (S is converted later)
        float* Xs = Mw + 64 * 64;                               // block products, up to 3 x [16][16]
        if (ok && warp < 2) {
            const int bi = tid >> 4, rr = tid & 15, i = 16 * bi + rr;
            float z[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) z[j] = (j == rr) ? 1.f : 0.f;
#pragma unroll
            for (int m = 15; m >= 1; --m) {
                const float zm = z[m];
                const float4* ar = (const float4*)(Ab + (16 * bi + m) * 64 + 16 * bi);
#pragma unroll
                for (int g4 = 0; 4 * g4 < m; ++g4) {
                    const float4 a = ar[g4];
                    if (4 * g4 + 0 < m) z[4 * g4 + 0] = fmaf(-zm, a.x, z[4 * g4 + 0]);
                    if (4 * g4 + 1 < m) z[4 * g4 + 1] = fmaf(-zm, a.y, z[4 * g4 + 1]);
                    if (4 * g4 + 2 < m) z[4 * g4 + 2] = fmaf(-zm, a.z, z[4 * g4 + 2]);
                    if (4 * g4 + 3 < m) z[4 * g4 + 3] = fmaf(-zm, a.w, z[4 * g4 + 3]);
                }
            }
            float* mrow = Mw + i * 64;
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const int c = 4 * c4;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if ((c >> 4) == bi) v = make_float4(z[c & 15], z[(c & 15) + 1], z[(c & 15) + 2], z[(c & 15) + 3]);
                *(float4*)(mrow + c) = v;
            }
        }
        __syncthreads();
        for (int d = 1; d <= 3; ++d) {
            const int ne = (4 - d) * 256;
            if (ok) {
                for (int e = tid; e < ne; e += kPcThreads) {
                    const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15, i = b + d, j = b;
                    const float* arow = Ab + (16 * i + r) * 64;
                    float acc = 0.f;
                    for (int kk = 16 * j; kk < 16 * i; kk += 4) {
                        const float4 a = *(const float4*)(arow + kk);
                        acc = fmaf(a.x, Mw[(kk + 0) * 64 + 16 * j + cc], acc);
                        acc = fmaf(a.y, Mw[(kk + 1) * 64 + 16 * j + cc], acc);
                        acc = fmaf(a.z, Mw[(kk + 2) * 64 + 16 * j + cc], acc);
                        acc = fmaf(a.w, Mw[(kk + 3) * 64 + 16 * j + cc], acc);
                    }
                    Xs[e] = acc;
                }
            }
            __syncthreads();
            if (ok) {
                for (int e = tid; e < ne; e += kPcThreads) {
                    const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15, i = b + d, j = b;
                    const float* drow = Mw + (16 * i + r) * 64 + 16 * i;
                    float acc = 0.f;
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) acc = fmaf(drow[kk], Xs[(b << 8) + (kk << 4) + cc], acc);
                    Mw[(16 * i + r) * 64 + 16 * j + cc] = -acc;
                }
            }
            __syncthreads();
        }
        if (ok && warp < 2) {
            // M row r -> TMEM R0 columns 64..127 (lane r); T = M Diag(beta) -> bf16 tile
            const int r = tid;
            const float* mrow = Mw + r * 64;
#pragma unroll
            for (int j = 0; j < 64; j += 16) {
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = mrow[j + e];
                tmem_st16(tmem_addr(R0, 32 * warp, 64 + j), f);
            }
            tmem_wait_st();
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                float t8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = mrow[j + e] * s_beta[j + e];
                *(uint4*)(sm + L::kTT + toff(r, j, 64)) = pk8(t8);
            }
        }
    }
    fence_proxy_async_smem();
    cta_sync();

    // ---- phase 3: W = T K~ (R1), U0 = T V (R2); U = U0 - W S (R2) ----
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R1, dk_(sm + L::kTT, ks, 64), dmn(sm + L::kKQ, ks, 16384), id, ks > 0);
        tma_done = mbar_wait(&bars[0], 0, kWait);
        if (tma_done) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(R2, dk_(sm + L::kTT, ks, 64), dmn(sm + L::kVT, ks, 8192), id, ks > 0);
        }
        mma_commit(&bars[1]);
    }
    if (ok) {
        // S -> bf16 tile (over the solve's scratch); dGamma_i = sum_j dS'_ij S_ij with
        // dS' from its bf16 tile (landed with the loads of phase 0).  Two threads per
        // row of S, 64 columns each, every load issued first.
        const int i = tid >> 1, c0 = 64 * (tid & 1);
        float4 x[16];
        if (S_src) {
            const float4* srs = (const float4*)(S_src + (size_t)i * kD + c0);
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = srs[j];
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const bool landed = mbar_wait(&bars[0], 0, kWait);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float f[8] = {x[2 * j].x, x[2 * j].y, x[2 * j].z, x[2 * j].w,
                                x[2 * j + 1].x, x[2 * j + 1].y, x[2 * j + 1].z, x[2 * j + 1].w};
            *(uint4*)(sm + L::kSS + toff(i, c0 + 8 * j, 128)) = pk8(f);
            float g8[8];
            unpk8(*(const uint4*)(sm + L::kDS + toff(i, c0 + 8 * j, 128)), g8);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(f[e], g8[e], acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if ((tid & 1) == 0) s_dgam[i] = acc;
        if (!landed) ok = false;
    }
    if (tid == 0 && !tma_done) ok = false;
    ok = mma_done(ok);
    if (ok && quarter < 2) {
        const int r = 32 * quarter + lane;
#pragma unroll
        for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R1, 32 * quarter, j), f);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) f[e] = -f[e];
            *(uint4*)(sm + L::kWU + toff(r, j, 64)) = pk8(&f[0]);
            *(uint4*)(sm + L::kWU + toff(r, j + 8, 64)) = pk8(&f[8]);
        }
    }
    fence_proxy_async_smem();
    cta_sync();
    if (tid == 0 && ok) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R2, dk_(sm + L::kWU, ks, 64), dmn(sm + L::kSS, ks, 16384), idesc_bf16(128, 128, 0, 1), 1);
        mma_commit(&bars[1]);
    }
    ok = mma_done(ok);
    if (ok && quarter < 2) {
        const int r = 32 * quarter + lane;
#pragma unroll
        for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R2, 32 * quarter, j), f);
            tmem_wait_ld();
            *(uint4*)(sm + L::kWU + toff(r, j, 64)) = pk8(&f[0]);
            *(uint4*)(sm + L::kWU + toff(r, j + 8, 64)) = pk8(&f[8]);
        }
    }
    fence_proxy_async_smem();
    cta_sync();

    // ---- phase 4: dU = K^end dS' + P^T dO (R1), dK^end = U dS'^T (R2);
    //      then [dO S^T; dU S^T] (R3) and dP = dO U^T (R1 columns 0..63) ----
    if (tid == 0 && ok) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R1, dk_(sm + L::kKE, ks, 64), dmn(sm + L::kDS, ks, 16384), idesc_bf16(128, 128, 0, 1),
                        ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R1, dmn(sm + L::kPT, ks, 8192), dmn(sm + L::kDD, ks, 16384), idesc_bf16(128, 128, 1, 1), 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R2, dk_(sm + L::kWU, ks, 64), dk_(sm + L::kDS, ks, 128), idesc_bf16(128, 128, 0, 0), ks > 0);
        mma_commit(&bars[1]);
    }
    ok = mma_done(ok);
    if (ok && quarter < 2) {
        const int r = 32 * quarter + lane;
#pragma unroll
        for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R1, 32 * quarter, j), f);
            tmem_wait_ld();
            *(uint4*)(sm + L::kDD + toff(64 + r, j, 128)) = pk8(&f[0]);
            *(uint4*)(sm + L::kDD + toff(64 + r, j + 8, 128)) = pk8(&f[8]);
        }
    }
    fence_proxy_async_smem();
    cta_sync();
    if (tid == 0 && ok) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R3, dk_(sm + L::kDD, ks, 128), dk_(sm + L::kSS, ks, 128), idesc_bf16(128, 128, 0, 0), ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R1, dk_(sm + L::kDD, ks, 128), dk_(sm + L::kWU, ks, 64), idesc_bf16(128, 64, 0, 0), ks > 0);
        mma_commit(&bars[1]);
    }
    ok = mma_done(ok);
    if (ok) {
        if (quarter >= 2) {
            // dW = -dU S^T -> bf16 tile (over S, read by the MMA above); then clear
            // these accumulator rows for dK~ = dG K^ + T^T dW
            const int r = 32 * (quarter - 2) + lane;
#pragma unroll
            for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
                float f[16];
                tmem_ld16(tmem_addr(R3, 32 * quarter, j), f);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = -f[e];
                *(uint4*)(sm + L::kDW + toff(r, j, 64)) = pk8(&f[0]);
                *(uint4*)(sm + L::kDW + toff(r, j + 8, 64)) = pk8(&f[8]);
                float zz[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) zz[e] = 0.f;
                tmem_st16(tmem_addr(R3, 32 * quarter, j), zz);
            }
            tmem_wait_st();
        } else {
            // dP = LowerIncl(dO U^T), rows of real tokens only
            const int r = 32 * quarter + lane;
#pragma unroll
            for (int j = 32 * hcol; j < 32 * hcol + 32; j += 16) {
                float f[16];
                tmem_ld16(tmem_addr(R1, 32 * quarter, j), f);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = (j + e <= r && r < len) ? f[e] : 0.f;
                *(uint4*)(sm + L::kDP + toff(r, j, 64)) = pk8(&f[0]);
                *(uint4*)(sm + L::kDP + toff(r, j + 8, 64)) = pk8(&f[8]);
            }
        }
    }
    fence_proxy_async_smem();
    cta_sync();

    // ---- phase 5: dT = dW K~^T + dU V^T (R1 columns 64..127); then, in fp32 on
    //      CUDA cores, X1 = dT T^T, dA = StrictLower(-M^T X1), dbeta, dG ----
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R1 + 64, dk_(sm + L::kDW, ks, 64), dk_(sm + L::kKQ, ks, 128), id, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(R1 + 64, dk_(sm + L::kDD + 8192, ks, 128), dk_(sm + L::kVT, ks, 64), id, 1);
        mma_commit(&bars[1]);
    }
    ok = mma_done(ok);
    float* DT = (float*)(sm + L::kDT);
    float* MM = (float*)(sm + L::kMM);
    float* MT = (float*)(sm + L::kMT);
    float* X1 = (float*)(sm + L::kX1);
    if (ok && quarter < 2) {
        const int r = 32 * quarter + lane;
#pragma unroll
        for (int j = 32 * hcol; j < 32 * hcol + 32; j += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R1, 32 * quarter, 64 + j), f);
            tmem_wait_ld();
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4)
                *(float4*)(DT + r * kLd + j + 4 * e4) = make_float4(f[4 * e4], f[4 * e4 + 1], f[4 * e4 + 2], f[4 * e4 + 3]);
        }
        if (hcol == 0) {
#pragma unroll
            for (int j = 0; j < 64; j += 16) {
                float f[16];
                tmem_ld16(tmem_addr(R0, 32 * quarter, 64 + j), f);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4)
                    *(float4*)(MM + r * kLd + j + 4 * e4) =
                        make_float4(f[4 * e4], f[4 * e4 + 1], f[4 * e4 + 2], f[4 * e4 + 3]);
#pragma unroll
                for (int e = 0; e < 16; ++e) MT[(j + e) * 64 + r] = f[e];
            }
        }
    }
    cta_sync();
    const int i0 = (tid >> 4) * 4, j0 = (tid & 15) * 4;
    if (ok) {
        // X1[i][j] = sum_k dT[i][k] T[j][k],  T[j][k] = M[j][k] beta_k
        float acc[4][4] = {};
        for (int kk = 0; kk < 64; ++kk) {
            const float4 t4 = *(const float4*)(MT + kk * 64 + j0);
            const float bk = s_beta[kk];
            const float tb[4] = {t4.x * bk, t4.y * bk, t4.z * bk, t4.w * bk};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float d = DT[(i0 + a) * kLd + kk];
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(d, tb[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
            *(float4*)(X1 + (i0 + a) * 64 + j0) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        if (tid < 64) {             // colsum(M o dT)_j
            const int j = tid;
            float s = 0.f;
            for (int i = 0; i < 64; ++i) s = fmaf(MT[j * 64 + i], DT[i * kLd + j], s);
            s_cs[j] = s;
        }
    }
    __syncthreads();
    if (ok) {
        // dA[i][j] = -sum_k M[k][i] X1[k][j] for j < i (written over dT)
        float acc[4][4] = {};
        for (int kk = 0; kk < 64; ++kk) {
            const float4 m4 = *(const float4*)(MM + kk * kLd + i0);
            const float4 x4 = *(const float4*)(X1 + kk * 64 + j0);
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w}, xv[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(mv[a], xv[b], acc[a][b]);
        }
        float* DA = DT;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = i0 + a;
            float v[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) v[b] = (j0 + b < i) ? -acc[a][b] : 0.f;
            // (every dT read above happened before the barrier)
            *(float4*)(DA + i * kLd + j0) = make_float4(v[0], v[1], v[2], v[3]);
            const float bi = s_beta[i];
            *(uint2*)(sm + L::kDG + toff(i, j0, 64)) = make_uint2(pk2(bi * v[0], bi * v[1]), pk2(bi * v[2], bi * v[3]));
        }
    }
    __syncthreads();
    if (ok && warp < 2) {
        // dbeta_i = colsum(M o dT)_i + sum_{j<i} G[i][j] dA[i][j]   (G from TMEM)
        const int i = tid;
        const float* DA = DT;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 64; j += 16) {
            float f[16];
            tmem_ld16(tmem_addr(R0, 32 * warp, j), f);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) s = fmaf(f[e], DA[i * kLd + j + e], s);
        }
        s_dbeta[i] = s_cs[i] + s;
    }
    fence_proxy_async_smem();
    cta_sync();

    // ---- phase 6: dQ~ = dO S^T + dP K^ and dK~ = dG K^ + T^T dW (R3);
    //      dK^ = dP^T Q~ + dG^T K~ (R1); dV = T^T dU (R0 rows 64..127) ----
    if (tid == 0 && ok) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R3, dk_(sm + L::kDP, ks, 128), dmn(sm + L::kKH, ks, 8192), idesc_bf16(128, 128, 0, 1), 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R3, dmn(sm + L::kZ0, ks, 8192), dmn(sm + L::kDW, ks, 8192), idesc_bf16(128, 128, 1, 1), 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R1, dmn(sm + L::kDP, ks, 8192), dmn(sm + L::kKQ + 8192, ks, 16384),
                        idesc_bf16(128, 128, 1, 1), ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R1, dmn(sm + L::kDG, ks, 8192), dmn(sm + L::kKQ, ks, 16384), idesc_bf16(128, 128, 1, 1), 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(R0, dmn(sm + L::kZ0, ks, 8192), dmn(sm + L::kDD + 8192, ks, 16384),
                        idesc_bf16(128, 128, 1, 1), ks > 0);
        mma_commit(&bars[1]);
    }
    // meanwhile: g again (log2 units), fp32 [64][128]
    float* gs = (float*)(sm + L::kG);
    {
        float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float gl2[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * R + i;
            float la[8];
            if (kScalarGate) {
#pragma unroll
                for (int e = 0; e < 8; ++e) la[e] = s_lg[r];
            } else {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < len) v = *(const uint4*)(log_alpha + base + (size_t)r * rs);
                unpk8(v, la);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) { s8[e] = fmaf(la[e], kL2e, s8[e]); gl2[i][e] = s8[e]; }
        }
        float4* part = (float4*)(sm + L::kPT) + (R * kD + 8 * C) / 4;
        part[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
        part[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
        __syncthreads();
        if (tid < kD) {
            float* pc = (float*)(sm + L::kPT) + tid;
            float acc = 0.f;
            for (int rg = 0; rg < 16; ++rg) { const float x = pc[rg * kD]; pc[rg * kD] = acc; acc += x; }
        }
        __syncthreads();
        const float* pp = (const float*)(sm + L::kPT) + R * kD + 8 * C;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * R + i;
            float gv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) gv[e] = pp[e] + gl2[i][e];
            *(float4*)(gs + r * kD + 8 * C) = make_float4(gv[0], gv[1], gv[2], gv[3]);
            *(float4*)(gs + r * kD + 8 * C + 4) = make_float4(gv[4], gv[5], gv[6], gv[7]);
        }
    }
    ok = mma_done(ok);

    // ---- phase 7: gradients of k, q, v, log alpha, beta ----
    constexpr int kLdK = 132;
    float* dkt = (float*)(sm + L::kDKT);           // dK~ fp32 [64][132]
    float* dgs = (float*)(sm + L::kSS);            // dg fp32 [64][128]
    float* kts = (float*)(sm + L::kKQ);            // dK^end o K^end fp32 [64][128] (over K~, Q~)
    if (ok && quarter >= 2) {
        const int r = 32 * (quarter - 2) + lane;
        const int64_t t = t0 + r;
#pragma unroll
        for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
            float f[16], v[16];
            tmem_ld16(tmem_addr(R3, 32 * quarter, j), f);
            tmem_ld16(tmem_addr(R0, 32 * quarter, j), v);
            tmem_wait_ld();
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4)
                *(float4*)(dkt + r * kLdK + j + 4 * e4) = make_float4(f[4 * e4], f[4 * e4 + 1], f[4 * e4 + 2], f[4 * e4 + 3]);
            if (r < len) {
                float* dst = dv + ((size_t)t * H + h) * kD + j;
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4)
                    *(float4*)(dst + 4 * e4) = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
            }
        }
    }
    cta_sync();
    if (ok && quarter < 2) {
        const int r = 32 * quarter + lane;
        const int64_t t = t0 + r;
        const bool in = r < len;
#pragma unroll 1
        for (int j = 64 * hcol; j < 64 * hcol + 64; j += 16) {
            float dQt[16], dKh[16], dKe[16];
            tmem_ld16(tmem_addr(R3, 32 * quarter, j), dQt);
            tmem_ld16(tmem_addr(R1, 32 * quarter, j), dKh);
            tmem_ld16(tmem_addr(R2, 32 * quarter, j), dKe);
            tmem_wait_ld();
            float kv[16], qv[16];
            {
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a, c2 = a, d2 = a;
                if (in) {
                    const size_t gi = ((size_t)t * H + h) * kD + j;
                    a = *(const uint4*)(k + gi);
                    b = *(const uint4*)(k + gi + 8);
                    c2 = *(const uint4*)(q + gi);
                    d2 = *(const uint4*)(q + gi + 8);
                }
                unpk8(a, kv); unpk8(b, kv + 8); unpk8(c2, qv); unpk8(d2, qv + 8);
            }
            float dkv[16], dqv[16], dgv[16], ktv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float g = gs[r * kD + j + e];
                const float e1 = ex2(g), e2 = ex2(-g), e3 = ex2(s_gC[j + e] - g);
                const float dKt = dkt[r * kLdK + j + e];
                const float a1 = dKt * e1, a2 = dKh[e] * e2, a3 = dKe[e] * e3, a4 = dQt[e] * e1;
                dkv[e] = a1 + a2 + a3;
                dqv[e] = a4;
                dgv[e] = kv[e] * (a1 - a2 - a3) + qv[e] * a4;
                ktv[e] = kv[e] * a3;                       // dK^end o K^end
            }
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                *(float4*)(dgs + r * kD + j + 4 * e4) = make_float4(dgv[4 * e4], dgv[4 * e4 + 1], dgv[4 * e4 + 2], dgv[4 * e4 + 3]);
                *(float4*)(kts + r * kD + j + 4 * e4) = make_float4(ktv[4 * e4], ktv[4 * e4 + 1], ktv[4 * e4 + 2], ktv[4 * e4 + 3]);
            }
            if (in) {
                float* pk = dk + ((size_t)t * H + h) * kD + j;
                float* pq = dq + ((size_t)t * H + h) * kD + j;
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    *(float4*)(pk + 4 * e4) = make_float4(dkv[4 * e4], dkv[4 * e4 + 1], dkv[4 * e4 + 2], dkv[4 * e4 + 3]);
                    *(float4*)(pq + 4 * e4) = make_float4(dqv[4 * e4], dqv[4 * e4 + 1], dqv[4 * e4 + 2], dqv[4 * e4 + 3]);
                }
            }
        }
    }
    cta_sync();
    if (ok && tid < kD) {
        // dlog alpha_r = sum_{r' >= r} dg_r' + colsum(dK^end o K^end) + dGamma Gamma, per channel
        const int ch = tid;
        float acc = s_dgam[ch] * ex2(s_gC[ch]);
        for (int r = 0; r < kChunk; ++r) acc += kts[r * kD + ch];     // (zero on padding rows)
        for (int r = len - 1; r >= 0; --r) {
            acc += dgs[r * kD + ch];
            if (kScalarGate) dgs[r * kD + ch] = acc;
            else dla[((size_t)(t0 + r) * H + h) * kD + ch] = acc;
        }
    }
    if (kScalarGate) __syncthreads();
    if (ok && tid < len) {
        const int r = tid;
        dbeta[(size_t)(t0 + r) * H + h] = s_dbeta[r];
        if (kScalarGate) {
            float s = 0.f;
            for (int ch = 0; ch < kD; ++ch) s += dgs[r * kD + ch];
            dla[(size_t)(t0 + r) * H + h] = s;
        }
    }
    if (!ok && tid == 0) record_status(hdr, KDA_ERR_TIMEOUT);
    if (tid == 0 && !tma_done) mbar_wait(&bars[0], 0, kWait);   // the loads have landed before exit
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void kda_tc_bwd_slots(int32_t* __restrict__ slot, int64_t n) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c < n) slot[c] = (int32_t)c;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Scratch of the tensor-core backward, in order: snapshot slot per chunk, the
// forward's records and segment scratch, every chunk's end state (fp32), every
// chunk's end-state gradient (a bf16 operand tile), and the forward's (unused)
// outputs.
struct TcBwdLayout {
    size_t slot, recs, extra, snaps, dsend, out, total;
};
static size_t al1k(size_t x) { return (x + 1023) / 1024 * 1024; }
static TcBwdLayout tc_bwd_layout(int N, int H, int64_t T, int64_t chunks_ub) {
    TcBwdLayout L;
    const size_t st = (size_t)kD * kD * sizeof(float);
    L.slot = 0;
    L.recs = al1k((size_t)chunks_ub * sizeof(int32_t));
    L.extra = al1k(L.recs + (size_t)chunks_ub * H * TcRec::kBytes);
    L.snaps = al1k(L.extra + tc_extra_bytes(N, H, T));
    L.dsend = al1k(L.snaps + (size_t)chunks_ub * H * st);
    L.out = al1k(L.dsend + (size_t)chunks_ub * H * (st / 2));
    L.total = al1k(L.out + (size_t)T * H * kD * 2);
    return L;
}

size_t backward_tc_bytes(int N, int H, int64_t T, int64_t chunks_ub) {
    return tc_bwd_layout(N, H, T, chunks_ub).total;
}

cudaError_t backward_tc_launch(const BackwardArgs& a, int64_t chunks_ub, void* region, cudaStream_t stream) {
    cudaError_t e;
    const TcBwdLayout L = tc_bwd_layout(a.N, a.H, a.T, chunks_ub);
    uint8_t* base = (uint8_t*)region;
    int32_t* slot = (int32_t*)(base + L.slot);
    float* snaps = (float*)(base + L.snaps);
    uint8_t* dsend = base + L.dsend;
    if (chunks_ub > 0) {
        kda_tc_bwd_slots<<<(unsigned)((chunks_ub + 255) / 256), 256, 0, stream>>>(slot, chunks_ub);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the forward, saving the state after every chunk
    PrefillArgs f;
    memset(&f, 0, sizeof(f));
    f.dtype = KDA_BF16; f.d = kD; f.N = a.N; f.H = a.H; f.chunks_ub = (int)chunks_ub; f.T = a.T;
    f.q = a.q; f.k = a.k; f.v = a.v; f.la = a.la; f.beta = a.beta; f.la_scalar = a.la_scalar;
    f.cu = a.cu; f.s0 = a.s0; f.out = base + L.out; f.sf = nullptr;
    f.hdr = a.hdr; f.chunk_first = a.chunk_first; f.recs = base + L.recs; f.extra = base + L.extra;
    f.phase_events = nullptr; f.snap_slot = slot; f.snaps = snaps;
    if ((e = prefill_tc_launch(f, a.T, stream)) != cudaSuccess) return e;

    RcArgs r;
    memset(&r, 0, sizeof(r));
    CUtensorMap tm_v, tm_do;
    memset(&tm_v, 0, sizeof(tm_v));
    memset(&tm_do, 0, sizeof(tm_do));
    if (a.T > 0) {
        if (!tc_make_tile_map(&tm_do, a.dout, a.T, a.H) || !tc_make_tile_map(&tm_v, a.v, a.T, a.H))
            return cudaErrorInvalidValue;
    }
    r.tm_do = tm_do;
    r.cu = a.cu; r.hdr = (DeviceHeader*)a.hdr; r.chunk_first = a.chunk_first; r.H = a.H;
    r.recs = base + L.recs; r.dfinal = a.dfinal; r.dsend = dsend; r.ds0 = a.ds0;
    if ((e = cudaFuncSetAttribute(kda_tc_bwd_chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)RcSmem::kBytes)) != cudaSuccess) return e;
    kda_tc_bwd_chain<<<(unsigned)a.N * a.H, kRcThreads, RcSmem::kBytes, stream>>>(r);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    if (chunks_ub > 0 && a.T > 0) {
        auto chunk = a.la_scalar ? kda_tc_bwd_chunk<true> : kda_tc_bwd_chunk<false>;
        if ((e = cudaFuncSetAttribute(chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)PcSmem::kBytes)) != cudaSuccess) return e;
        chunk<<<dim3((unsigned)chunks_ub, a.H), kPcThreads, PcSmem::kBytes, stream>>>(
            tm_v, tm_do, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.la,
            (const __nv_bfloat16*)a.beta, a.cu, (DeviceHeader*)a.hdr, a.chunk_first, a.N, a.H, a.s0, snaps, dsend,
            a.dq, a.dk, a.dv, a.dla, a.dbeta);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda

// kda_prefill_simt.cu -- chunk-parallel KDA prefill on CUDA cores, all fp32.
//
// This is the path for fp32 inputs (and for any shape the tensor-core path
// does not take).  Every product is an fp32 FMA with fp32 accumulation, so
// its only error is fp32 rounding.
//
// Chunk algebra ("Kimi Delta Attention" deep dive, section 06: matrix
// products inside a chunk, only the boundary state carried between chunks;
// derived from the recurrence of section 03).  For a chunk of C tokens with
// start state S0, g_r = sum_{i<=r} log alpha_i per key channel:
//
//   A[i][j] = beta_i sum_c k_ic k_jc exp(g_ic - g_jc)   (j < i)
//   P[i][j] =        sum_c q_ic k_jc exp(g_ic - g_jc)   (j <= i)
//   T = (I + A)^-1 Diag(beta)
//   W = T K~,  U0 = T V          K~ = K * exp(g)
//   Q' = Q~ - P W,  O0 = P U0    Q~ = Q * exp(g)
//   K^end = K * exp(g_C - g),  Gamma = exp(g_C)
//
// and, carried across the chunks of one sequence in order (kernel b):
//
//   U = U0 - W S,   O = O0 + Q' S,   S <- Diag(Gamma) S + K^end^T U.
//
// Every exponent above is <= 0 for log alpha <= 0 (i >= j inside A and P),
// so nothing overflows however strong the decay.
#include "kda_common.cuh"
#include "kda_paths.h"

namespace kda {

constexpr int kSimtThreads = 256;
constexpr int kSimtTile = 32;                  // state columns per CTA in kernel (b)

// Workspace record per (chunk, head): W, Q', K^end, U0, O0 [C x D] then Gamma [D], fp32.
template <int D> struct SimtRec {
    static constexpr size_t kW = 0, kQp = (size_t)kChunk * D, kKe = 2 * (size_t)kChunk * D,
                            kU0 = 3 * (size_t)kChunk * D, kO0 = 4 * (size_t)kChunk * D,
                            kG = 5 * (size_t)kChunk * D, kFloats = 5 * (size_t)kChunk * D + D;
};

size_t simt_record_bytes(int d) { return (5 * (size_t)kChunk * d + d) * sizeof(float); }

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
kda_simt_intra_chunk(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ log_alpha, int la_scalar, const T* __restrict__ beta,
                     const int32_t* __restrict__ cu, const DeviceHeader* __restrict__ hdr,
                     const int32_t* __restrict__ chunk_first, int N, int H, float* __restrict__ ws) {
    if (hdr->status != KDA_OK) return;
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= hdr->total_chunks) return;
    const int n = chunk_owner(chunk_first, N, c);
    const int64_t t0 = (int64_t)cu[n] + (int64_t)(c - chunk_first[n]) * kChunk;
    const int len = (int)min64(kChunk, (int64_t)cu[n + 1] - t0);

    extern __shared__ float smem[];
    constexpr int LDP = kChunk + 1;            // padded row of the C x C matrices
    float* Ks = smem;                          // [C][D]  K, then K~, then U0
    float* Qs = Ks + kChunk * D;               // [C][D]  Q, then Q~
    float* Vs = Qs + kChunk * D;               // [C][D]  V
    float* Gs = Vs + kChunk * D;               // [C][D]  g, then W
    float* As = Gs + kChunk * D;               // [C][LDP] A
    float* Ps = As + kChunk * LDP;             // [C][LDP] P
    float* Xs = Ps + kChunk * LDP;             // [C][LDP] (I+A)^-1, then T
    float* bs = Xs + kChunk * LDP;             // [C] beta
    float* gC = bs + kChunk;                   // [D] g at the last token of the chunk
    const int tid = threadIdx.x;

    for (int e = tid; e < kChunk * D; e += kSimtThreads) {
        const int r = e / D, ch = e % D;
        const bool ok = r < len;
        const size_t gi = ((size_t)(t0 + r) * H + h) * D + ch;
        Ks[e] = ok ? to_f32(k[gi]) : 0.f;
        Qs[e] = ok ? to_f32(q[gi]) : 0.f;
        Vs[e] = ok ? to_f32(v[gi]) : 0.f;
        Gs[e] = ok ? to_f32(log_alpha[la_scalar ? (size_t)(t0 + r) * H + h : gi]) : 0.f;
    }
    if (tid < kChunk) bs[tid] = tid < len ? to_f32(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    __syncthreads();
    if (tid < D) {                              // g = inclusive cumsum of log alpha, per channel
        float g = 0.f;
        for (int r = 0; r < kChunk; ++r) { g += Gs[r * D + tid]; Gs[r * D + tid] = g; }
        gC[tid] = g;
    }
    __syncthreads();

    // A (strictly lower, scaled by beta_i) and P (lower incl. diagonal).
    for (int e = tid; e < kChunk * kChunk; e += kSimtThreads) {
        const int i = e / kChunk, j = e % kChunk;
        float a = 0.f, p = 0.f;
        if (j <= i) {
            const float* ki = Ks + i * D; const float* kj = Ks + j * D; const float* qi = Qs + i * D;
            const float* gi = Gs + i * D; const float* gj = Gs + j * D;
            for (int ch = 0; ch < D; ++ch) {
                const float ek = kj[ch] * expf(gi[ch] - gj[ch]);
                a += ki[ch] * ek;
                p += qi[ch] * ek;
            }
        }
        As[i * LDP + j] = j < i ? bs[i] * a : 0.f;
        Ps[i * LDP + j] = p;
    }
    __syncthreads();

    // (I + A)^-1 by forward substitution, one column per thread.
    if (tid < kChunk) {
        const int j = tid;
        for (int i = 0; i < kChunk; ++i) {
            float x = (i == j) ? 1.f : 0.f;
            if (i > j) {
                for (int m = j; m < i; ++m) x -= As[i * LDP + m] * Xs[m * LDP + j];
            }
            Xs[i * LDP + j] = x;
        }
    }
    __syncthreads();

    // T = X Diag(beta); K^end out; K~ and Q~ in place.
    float* rec = ws + ((size_t)c * H + h) * SimtRec<D>::kFloats;
    for (int e = tid; e < kChunk * kChunk; e += kSimtThreads) {
        const int i = e / kChunk, j = e % kChunk;
        Xs[i * LDP + j] *= bs[j];
    }
    for (int e = tid; e < kChunk * D; e += kSimtThreads) {
        const int ch = e % D;
        const float g = Gs[e];
        rec[SimtRec<D>::kKe + e] = Ks[e] * expf(gC[ch] - g);
        const float eg = expf(g);
        Ks[e] *= eg;
        Qs[e] *= eg;
    }
    if (tid < D) rec[SimtRec<D>::kG + tid] = expf(gC[tid]);
    __syncthreads();

    // W = T K~ -> Gs (g no longer needed), then U0 = T V -> Ks (K~ no longer needed).
    for (int e = tid; e < kChunk * D; e += kSimtThreads) {
        const int i = e / D, ch = e % D;
        float w = 0.f;
        for (int m = 0; m <= i; ++m) w += Xs[i * LDP + m] * Ks[m * D + ch];
        Gs[e] = w;
        rec[SimtRec<D>::kW + e] = w;
    }
    __syncthreads();
    for (int e = tid; e < kChunk * D; e += kSimtThreads) {
        const int i = e / D, ch = e % D;
        float u = 0.f;
        for (int m = 0; m <= i; ++m) u += Xs[i * LDP + m] * Vs[m * D + ch];
        Ks[e] = u;
        rec[SimtRec<D>::kU0 + e] = u;
    }
    __syncthreads();
    // Q' = Q~ - P W,  O0 = P U0.
    for (int e = tid; e < kChunk * D; e += kSimtThreads) {
        const int i = e / D, ch = e % D;
        float pw = 0.f, pu = 0.f;
        for (int m = 0; m <= i; ++m) {
            const float p = Ps[i * LDP + m];
            pw += p * Gs[m * D + ch];
            pu += p * Ks[m * D + ch];
        }
        rec[SimtRec<D>::kQp + e] = Qs[e] - pw;
        rec[SimtRec<D>::kO0 + e] = pu;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
kda_simt_inter_chunk(const int32_t* __restrict__ cu, const DeviceHeader* __restrict__ hdr,
                     const int32_t* __restrict__ chunk_first, int H,
                     const float* __restrict__ ws, const float* __restrict__ initial_state,
                     T* __restrict__ out, float* __restrict__ final_state,
                     const int32_t* __restrict__ snap_slot, float* __restrict__ snaps) {
    if (hdr->status != KDA_OK) return;
    const int nh = blockIdx.x;
    const int n = nh / H, h = nh % H;
    const int col0 = blockIdx.y * kSimtTile;
    extern __shared__ float smem[];
    float* Wsm = smem;                          // [C][D]
    float* Qsm = Wsm + kChunk * D;              // [C][D]
    float* Esm = Qsm + kChunk * D;              // [C][D]  K^end
    float* Ssm = Esm + kChunk * D;              // [D][32] state tile
    float* Usm = Ssm + D * kSimtTile;           // [C][32]
    float* Gsm = Usm + kChunk * kSimtTile;      // [D]
    const int tid = threadIdx.x;
    const int j = tid % kSimtTile, r0 = tid / kSimtTile;   // 8 row groups

    const size_t sbase = (size_t)nh * D * D;
    for (int e = tid; e < D * kSimtTile; e += kSimtThreads) {
        const int r = e / kSimtTile, cc = e % kSimtTile;
        Ssm[e] = initial_state ? initial_state[sbase + (size_t)r * D + col0 + cc] : 0.f;
    }
    const int64_t seq0 = cu[n];
    const int c_begin = chunk_first[n], c_end = chunk_first[n + 1];
    for (int c = c_begin; c < c_end; ++c) {
        const float* rec = ws + ((size_t)c * H + h) * SimtRec<D>::kFloats;
        const int64_t t0 = seq0 + (int64_t)(c - c_begin) * kChunk;
        const int len = (int)min64(kChunk, (int64_t)cu[n + 1] - t0);
        __syncthreads();                        // previous chunk done with the buffers
        for (int e = tid; e < kChunk * D; e += kSimtThreads) {
            Wsm[e] = rec[SimtRec<D>::kW + e];
            Qsm[e] = rec[SimtRec<D>::kQp + e];
            Esm[e] = rec[SimtRec<D>::kKe + e];
        }
        if (tid < D) Gsm[tid] = rec[SimtRec<D>::kG + tid];
        __syncthreads();
        // U = U0 - W S and O = O0 + Q' S for this column tile.
        for (int i = r0; i < kChunk; i += kSimtThreads / kSimtTile) {
            float ws_ = 0.f, qs_ = 0.f;
            for (int ch = 0; ch < D; ++ch) {
                const float s = Ssm[ch * kSimtTile + j];
                ws_ += Wsm[i * D + ch] * s;
                qs_ += Qsm[i * D + ch] * s;
            }
            Usm[i * kSimtTile + j] = rec[SimtRec<D>::kU0 + (size_t)i * D + col0 + j] - ws_;
            if (i < len)
                out[((size_t)(t0 + i) * H + h) * D + col0 + j] =
                    from_f32<T>(rec[SimtRec<D>::kO0 + (size_t)i * D + col0 + j] + qs_);
        }
        __syncthreads();
        // S <- Diag(Gamma) S + K^end^T U; written out too if a snapshot is
        // requested after this chunk.
        const int snap_m = snap_slot ? snap_slot[c] : -1;
        for (int ch = r0; ch < D; ch += kSimtThreads / kSimtTile) {
            float acc = Gsm[ch] * Ssm[ch * kSimtTile + j];
            for (int i = 0; i < kChunk; ++i) acc += Esm[i * D + ch] * Usm[i * kSimtTile + j];
            Ssm[ch * kSimtTile + j] = acc;
            if (snap_m >= 0) snaps[(((size_t)snap_m * H + h) * D + ch) * D + col0 + j] = acc;
        }
    }
    __syncthreads();
    if (final_state)
        for (int e = tid; e < D * kSimtTile; e += kSimtThreads) {
            const int r = e / kSimtTile, cc = e % kSimtTile;
            final_state[sbase + (size_t)r * D + col0 + cc] = Ssm[e];
        }
}

template <typename T, int D>
static cudaError_t launch_simt(const PrefillArgs& a, cudaStream_t stream) {
    constexpr int LDP = kChunk + 1;
    const size_t smem_a = (4 * (size_t)kChunk * D + 3 * (size_t)kChunk * LDP + kChunk + D) * sizeof(float);
    const size_t smem_b = (3 * (size_t)kChunk * D + (size_t)D * kSimtTile + kChunk * kSimtTile + D) * sizeof(float);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(kda_simt_intra_chunk<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_a)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kda_simt_inter_chunk<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_b)) != cudaSuccess) return e;
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[0], stream)) != cudaSuccess) return e;
    if (a.chunks_ub > 0) {
        kda_simt_intra_chunk<T, D><<<dim3(a.chunks_ub, a.H), kSimtThreads, smem_a, stream>>>(
            (const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.la, a.la_scalar, (const T*)a.beta, a.cu,
            (const DeviceHeader*)a.hdr, a.chunk_first, a.N, a.H, (float*)a.recs);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[1], stream)) != cudaSuccess) return e;
    kda_simt_inter_chunk<T, D><<<dim3((unsigned)a.N * a.H, D / kSimtTile), kSimtThreads, smem_b, stream>>>(
        a.cu, (const DeviceHeader*)a.hdr, a.chunk_first, a.H, (const float*)a.recs, a.s0, (T*)a.out, a.sf,
        a.snap_slot, a.snaps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.phase_events && (e = cudaEventRecord(a.phase_events[2], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t prefill_simt_launch(const PrefillArgs& a, cudaStream_t stream) {
    if (a.dtype == KDA_BF16)
        return a.d == 128 ? launch_simt<__nv_bfloat16, 128>(a, stream) : launch_simt<__nv_bfloat16, 64>(a, stream);
    return a.d == 128 ? launch_simt<float, 128>(a, stream) : launch_simt<float, 64>(a, stream);
}

}  // namespace kda

// kda_backward.cu -- reverse mode (gradients) of the KDA prefill, fp32 on
// CUDA cores.
//
// Per sequence and head, with S' = Diag(alpha_t) S_{t-1}, e = v_t - S'^T k_t,
// S_t = S' + beta_t k_t e^T and o_t = S_t^T q_t (the recurrence of the "Kimi
// Delta Attention" deep dive, section 03, read as in section 02), and dS the
// gradient of the loss with respect to S_t, token t contributes, in reverse
// order:
//
//   read:   dq_t = S_t do_t;                 dS += q_t do_t^T
//   write:  u = dS^T k_t;  de = beta_t u;    dbeta_t = e . u;   dv_t = de
//           dk_t = beta_t dS e - S' de;      dS' = dS - k_t de^T
//   decay:  dlog_alpha_t = alpha_t o rowsum(dS' o S_{t-1});     dS <- Diag(alpha_t) dS'
//
// Columns of S (and of dS) never mix, so a CTA owns a 32-column tile of one
// (sequence, head) and walks the whole sequence: first forward, keeping the
// tile's state every kBlk tokens in the workspace, then backwards block by
// block, recomputing the block's states into shared memory and applying the
// rules above.  dv and the initial-state gradient belong to the tile; dq, dk,
// dlog_alpha and dbeta are sums over all columns, so each tile writes its
// partial sums and a second kernel adds the tiles in a fixed order (no
// atomics: the result is deterministic).
#include "kda_common.cuh"
#include "kda_paths.h"

namespace kda {

constexpr int kBwdCols = 32;        // state columns per CTA
constexpr int kBwdThreads = 256;    // 8 row groups x 32 columns
constexpr int kBlk = 8;             // tokens between kept states

template <int D> struct BwdSmem {
    static constexpr int kRP = D / 8;                 // rows per thread
    float st[kBlk][D][kBwdCols];                      // S_{t-1} of each token of the block
    float k[kBlk][D], q[kBlk][D], alpha[kBlk][D];
    float e[kBlk][kBwdCols], v[kBlk][kBwdCols], dout[kBlk][kBwdCols];
    float beta[kBlk];
    float red_rows[8][kBwdCols];                      // per-row-group partial column sums
    float red_cols[3][D][kBwdCols + 1];               // per-column partials of dq, dk, dalpha
};

// Loads the per-token inputs of tokens [t, t + n) of head h into shared memory.
template <typename T, int D>
__device__ __forceinline__ void bwd_load_tokens(BwdSmem<D>& sm, int64_t t, int n, int h, int H, int col0,
                                                const T* q, const T* k, const T* v, const T* la, int la_scalar,
                                                const T* beta, const T* dout) {
    for (int e = threadIdx.x; e < n * D; e += kBwdThreads) {
        const int r = e / D, i = e % D;
        const size_t gi = ((size_t)(t + r) * H + h) * D + i;
        sm.k[r][i] = to_f32(k[gi]);
        sm.q[r][i] = to_f32(q[gi]);
        sm.alpha[r][i] = expf(to_f32(la[la_scalar ? (size_t)(t + r) * H + h : gi]));
    }
    for (int e = threadIdx.x; e < n * kBwdCols; e += kBwdThreads) {
        const int r = e / kBwdCols, j = e % kBwdCols;
        const size_t gi = ((size_t)(t + r) * H + h) * D + col0 + j;
        sm.v[r][j] = to_f32(v[gi]);
        sm.dout[r][j] = to_f32(dout[gi]);
    }
    if (threadIdx.x < n) sm.beta[threadIdx.x] = to_f32(beta[(size_t)(t + threadIdx.x) * H + h]);
}

// One forward step on the thread's rows of column j: S <- S' + beta k e^T,
// with the column sum over row groups through red_rows.  Returns e_j.
template <int D>
__device__ __forceinline__ float bwd_fwd_step(BwdSmem<D>& sm, float (&S)[D / 8], int r, int rg, int j) {
    constexpr int RP = D / 8;
    float pk = 0.f;
#pragma unroll
    for (int a = 0; a < RP; ++a) {
        const int i = rg * RP + a;
        S[a] *= sm.alpha[r][i];
        pk = fmaf(sm.k[r][i], S[a], pk);
    }
    sm.red_rows[rg][j] = pk;
    __syncthreads();
    float pred = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) pred += sm.red_rows[g][j];
    const float e = sm.v[r][j] - pred;
    const float be = sm.beta[r] * e;
#pragma unroll
    for (int a = 0; a < RP; ++a) S[a] = fmaf(sm.k[r][rg * RP + a], be, S[a]);
    __syncthreads();                                   // red_rows free again
    return e;
}

template <typename T, int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
kda_backward_tile(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const T* __restrict__ la, int la_scalar, const T* __restrict__ beta,
                  const int32_t* __restrict__ cu, const DeviceHeader* __restrict__ hdr,
                  const int32_t* __restrict__ chunk_first, int H, int64_t T_tot,
                  const float* __restrict__ s0, const T* __restrict__ dout, const float* __restrict__ dfinal,
                  float* __restrict__ ckpt, float* __restrict__ part, float* __restrict__ dv,
                  float* __restrict__ ds0) {
    constexpr int RP = D / 8;
    constexpr int kTiles = D / kBwdCols;
    if (hdr->status != KDA_OK) return;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
    const int nh = blockIdx.x, tile = blockIdx.y, n = nh / H, h = nh % H;
    const int col0 = tile * kBwdCols;
    const int tid = threadIdx.x, rg = tid >> 5, j = tid & 31;
    const int64_t t0 = cu[n];
    const int L = (int)(cu[n + 1] - t0);
    // kept states: block b of this sequence at ckpt[((blk0 + b) * H + h) * kTiles + tile]
    const int64_t blk0 = (int64_t)chunk_first[n] * (kChunk / kBlk);
    auto kept = [&](int b) { return ckpt + (((size_t)(blk0 + b) * H + h) * kTiles + tile) * (size_t)D * kBwdCols; };
    const size_t sbase = (size_t)nh * D * D;

    // ---- forward: keep the state at the start of every block
    float S[RP];
#pragma unroll
    for (int a = 0; a < RP; ++a) S[a] = s0 ? s0[sbase + (size_t)(rg * RP + a) * D + col0 + j] : 0.f;
    for (int b = 0; b * kBlk < L; ++b) {
        float* kp = kept(b);
#pragma unroll
        for (int a = 0; a < RP; ++a) kp[(rg * RP + a) * kBwdCols + j] = S[a];
        const int n_b = min(kBlk, L - b * kBlk);
        __syncthreads();
        bwd_load_tokens<T, D>(sm, t0 + (int64_t)b * kBlk, n_b, h, H, col0, q, k, v, la, la_scalar, beta, dout);
        __syncthreads();
        for (int r = 0; r < n_b; ++r) bwd_fwd_step<D>(sm, S, r, rg, j);
    }

    // ---- backward, block by block from the end
    float dS[RP];
#pragma unroll
    for (int a = 0; a < RP; ++a) dS[a] = dfinal ? dfinal[sbase + (size_t)(rg * RP + a) * D + col0 + j] : 0.f;
    const int nblk = (L + kBlk - 1) / kBlk;
    for (int b = nblk - 1; b >= 0; --b) {
        const int n_b = min(kBlk, L - b * kBlk);
        const int64_t tb = t0 + (int64_t)b * kBlk;
        __syncthreads();
        bwd_load_tokens<T, D>(sm, tb, n_b, h, H, col0, q, k, v, la, la_scalar, beta, dout);
        const float* kp = kept(b);
#pragma unroll
        for (int a = 0; a < RP; ++a) S[a] = kp[(rg * RP + a) * kBwdCols + j];
        __syncthreads();
        // recompute the block: st[r] = S_{t-1} of token r, e[r]
        for (int r = 0; r < n_b; ++r) {
#pragma unroll
            for (int a = 0; a < RP; ++a) sm.st[r][rg * RP + a][j] = S[a];
            const float e = bwd_fwd_step<D>(sm, S, r, rg, j);
            if (rg == 0) sm.e[r][j] = e;
        }
        __syncthreads();
        for (int r = n_b - 1; r >= 0; --r) {
            const int64_t t = tb + r;
            const float bt = sm.beta[r], e_j = sm.e[r][j], do_j = sm.dout[r][j];
            float Sp[RP], Sprev[RP];
            float pq[RP], pk[RP], pa[RP];
            // read: dq = S_t do, dS += q do^T
            float uk = 0.f;
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const int i = rg * RP + a;
                Sprev[a] = sm.st[r][i][j];
                Sp[a] = sm.alpha[r][i] * Sprev[a];
                const float St = fmaf(sm.k[r][i], bt * e_j, Sp[a]);
                pq[a] = St * do_j;
                dS[a] = fmaf(sm.q[r][i], do_j, dS[a]);
                uk = fmaf(sm.k[r][i], dS[a], uk);
            }
            sm.red_rows[rg][j] = uk;
            __syncthreads();
            float u = 0.f;
#pragma unroll
            for (int g = 0; g < 8; ++g) u += sm.red_rows[g][j];
            const float de = bt * u;
            if (rg == 0) dv[((size_t)t * H + h) * D + col0 + j] = de;
            // write and decay
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const int i = rg * RP + a;
                pk[a] = bt * dS[a] * e_j - Sp[a] * de;
                const float dSp = fmaf(-sm.k[r][i], de, dS[a]);
                pa[a] = dSp * Sprev[a];
                dS[a] = sm.alpha[r][i] * dSp;
            }
            // column sums of dq, dk, dalpha over the tile: transpose through shared memory
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const int i = rg * RP + a;
                sm.red_cols[0][i][j] = pq[a];
                sm.red_cols[1][i][j] = pk[a];
                sm.red_cols[2][i][j] = pa[a];
            }
            __syncthreads();
            // dbeta partial = e . u over the tile (u_j of every column is in red_rows)
            float* pt = part + ((size_t)tile * T_tot + t) * H * (3 * D + 1) + (size_t)h * (3 * D + 1);
            for (int w = tid; w < 3 * D; w += kBwdThreads) {
                const int m = w / D, i = w % D;
                float acc = 0.f;
#pragma unroll 8
                for (int c = 0; c < kBwdCols; ++c) acc += sm.red_cols[m][i][c];
                pt[w] = m == 2 ? acc * sm.alpha[r][i] : acc;
            }
            if (tid < 32) {
                float eu = 0.f;
                for (int g = 0; g < 8; ++g) eu += sm.red_rows[g][tid];   // u of column tid
                eu *= sm.e[r][tid];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) eu += __shfl_xor_sync(0xffffffffu, eu, o);
                if (tid == 0) pt[3 * D] = eu;
            }
            __syncthreads();
        }
    }
    if (ds0) {
#pragma unroll
        for (int a = 0; a < RP; ++a) ds0[sbase + (size_t)(rg * RP + a) * D + col0 + j] = dS[a];
    }
}

// Adds the tiles' partial sums: dq, dk, dlog_alpha (per channel, or summed
// over channels for a scalar gate) and dbeta, in tile order.
template <int D>
__global__ void __launch_bounds__(256)
kda_backward_reduce(const float* __restrict__ part, const DeviceHeader* __restrict__ hdr, int64_t T_tot, int H,
                    int la_scalar, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dla,
                    float* __restrict__ dbeta) {
    constexpr int kTiles = D / kBwdCols;
    constexpr int W = 3 * D + 1;
    if (hdr->status != KDA_OK) return;
    const int64_t th = blockIdx.x;                    // (token, head)
    if (th >= T_tot * H) return;
    __shared__ float s_la[D];
    for (int w = threadIdx.x; w < W; w += blockDim.x) {
        float acc = 0.f;
        for (int tl = 0; tl < kTiles; ++tl) acc += part[((size_t)tl * T_tot * H + th) * W + w];
        const int m = w / D, i = w % D;
        if (w == 3 * D) dbeta[th] = acc;
        else if (m == 0) dq[th * D + i] = acc;
        else if (m == 1) dk[th * D + i] = acc;
        else if (la_scalar) s_la[i] = acc;
        else dla[th * D + i] = acc;
    }
    if (la_scalar) {
        __syncthreads();
        if (threadIdx.x < 32) {
            float a = 0.f;
            for (int i = threadIdx.x; i < D; i += 32) a += s_la[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (threadIdx.x == 0) dla[th] = a;
        }
    }
}

size_t backward_ckpt_bytes(int d, int H, int64_t chunks_ub) {
    return (size_t)chunks_ub * (kChunk / kBlk) * H * (size_t)d * d * sizeof(float);
}
size_t backward_part_bytes(int d, int H, int64_t T) {
    return (size_t)(d / kBwdCols) * T * H * (3 * (size_t)d + 1) * sizeof(float);
}

template <typename T, int D>
static cudaError_t launch_bwd(const BackwardArgs& a, cudaStream_t stream) {
    cudaError_t e;
    const size_t smem = sizeof(BwdSmem<D>);
    if ((e = cudaFuncSetAttribute(kda_backward_tile<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess) return e;
    kda_backward_tile<T, D><<<dim3((unsigned)a.N * a.H, D / kBwdCols), kBwdThreads, smem, stream>>>(
        (const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.la, a.la_scalar, (const T*)a.beta, a.cu,
        (const DeviceHeader*)a.hdr, a.chunk_first, a.H, a.T, a.s0, (const T*)a.dout, a.dfinal, a.ckpt, a.part,
        a.dv, a.ds0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.T > 0) {
        kda_backward_reduce<D><<<(unsigned)(a.T * a.H), 256, 0, stream>>>(
            a.part, (const DeviceHeader*)a.hdr, a.T, a.H, a.la_scalar, a.dq, a.dk, a.dla, a.dbeta);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t backward_launch(const BackwardArgs& a, cudaStream_t stream) {
    if (a.dtype == KDA_BF16)
        return a.d == 128 ? launch_bwd<__nv_bfloat16, 128>(a, stream) : launch_bwd<__nv_bfloat16, 64>(a, stream);
    return a.d == 128 ? launch_bwd<float, 128>(a, stream) : launch_bwd<float, 64>(a, stream);
}

}  // namespace kda

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
// Columns of S (and of dS) never mix, so a CTA owns a tile of 8, 16 or 32
// state columns of one (sequence, head) (the widest that still gives every SM
// a CTA) and walks the whole sequence: first forward, keeping the
// tile's state every kBlk tokens in the workspace, then backwards block by
// block, recomputing the block's states into shared memory and applying the
// rules above.  dv and the initial-state gradient belong to the tile; dq, dk,
// dlog_alpha and dbeta are sums over all columns, so each tile writes its
// partial sums and a second kernel adds the tiles in a fixed order (no
// atomics: the result is deterministic).
//
// This is the backward for fp32 inputs and head size 64, and the fallback of
// the tensor-core backward (kda_backward_tc.cu) for calls where some chunk's
// decay is too strong for the factorised chunk products: there it is launched
// after the tensor-core kernels and runs only if the forward flagged such a
// chunk (only_if_slow).
#include "kda_common.cuh"
#include "kda_paths.h"

namespace kda {

constexpr int kBwdThreads = 256;    // (256 / COLS) row groups x COLS columns
constexpr int kBlk = 8;             // tokens between kept states

// Thread (rg, j) = (tid % RG, tid / RG) owns rows i = a * RG + rg (a < RP) of
// column j: the RG row groups of a column sit in one warp, so sums over rows
// are warp shuffles, and neighbouring lanes touch neighbouring rows (shared
// memory without bank conflicts); sums over the tile's columns combine the
// warp's columns by shuffles and the 8 warps through red[].
template <int D, int COLS> struct BwdSmem {
    static constexpr int kRG = kBwdThreads / COLS;    // row groups (32, 16 or 8: a power of two <= 32)
    static constexpr int kRP = D / kRG;               // rows per thread
    float st[kBlk][kRP][COLS][kRG];                   // S_{t-1} of each token of the block, [.][a][j][rg]
    float k[kBlk][D], q[kBlk][D], alpha[kBlk][D];
    float e[kBlk][COLS], v[kBlk][COLS], dout[kBlk][COLS];
    float beta[kBlk];
    float red[2][kBwdThreads / 32][3 * D + 1];        // per-warp column sums (dq, dk, dalpha, dbeta), 2 buffers
};

// Sum over the RG lanes of a column (aligned lane groups of a warp).
template <int RG> __device__ __forceinline__ float rows_sum(float x) {
#pragma unroll
    for (int o = RG / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// Sum over the warp's columns (lanes RG apart).
template <int RG> __device__ __forceinline__ float warp_cols_sum(float x) {
#pragma unroll
    for (int o = RG; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Loads the per-token inputs of tokens [t, t + n) of head h into shared memory.
template <typename T, int D, int COLS>
__device__ __forceinline__ void bwd_load_tokens(BwdSmem<D, COLS>& sm, int64_t t, int n, int h, int H, int col0,
                                                const T* q, const T* k, const T* v, const T* la, int la_scalar,
                                                const T* beta, const T* dout) {
    for (int e = threadIdx.x; e < n * D; e += kBwdThreads) {
        const int r = e / D, i = e % D;
        const size_t gi = ((size_t)(t + r) * H + h) * D + i;
        sm.k[r][i] = to_f32(k[gi]);
        sm.q[r][i] = to_f32(q[gi]);
        sm.alpha[r][i] = expf(to_f32(la[la_scalar ? (size_t)(t + r) * H + h : gi]));
    }
    for (int e = threadIdx.x; e < n * COLS; e += kBwdThreads) {
        const int r = e / COLS, j = e % COLS;
        const size_t gi = ((size_t)(t + r) * H + h) * D + col0 + j;
        sm.v[r][j] = to_f32(v[gi]);
        sm.dout[r][j] = to_f32(dout[gi]);
    }
    if (threadIdx.x < n) sm.beta[threadIdx.x] = to_f32(beta[(size_t)(t + threadIdx.x) * H + h]);
}

// True on the lanes of a warp's first column (they hold the warp's column sums).
__device__ __forceinline__ bool lane_col0(int tid, int RG) { return (tid & 31) < RG; }

// One forward step on the thread's rows of column j: S <- S' + beta k e^T.
// Returns e_j.
template <int D, int COLS>
__device__ __forceinline__ float bwd_fwd_step(const BwdSmem<D, COLS>& sm, float (&S)[BwdSmem<D, COLS>::kRP],
                                              int r, int rg, int j) {
    constexpr int RP = BwdSmem<D, COLS>::kRP, RG = BwdSmem<D, COLS>::kRG;
    float pk = 0.f;
#pragma unroll
    for (int a = 0; a < RP; ++a) {
        const int i = a * RG + rg;
        S[a] *= sm.alpha[r][i];
        pk = fmaf(sm.k[r][i], S[a], pk);
    }
    const float e = sm.v[r][j] - rows_sum<RG>(pk);
    const float be = sm.beta[r] * e;
#pragma unroll
    for (int a = 0; a < RP; ++a) S[a] = fmaf(sm.k[r][a * RG + rg], be, S[a]);
    return e;
}

template <typename T, int D, int COLS>
__global__ void __launch_bounds__(kBwdThreads, 1)
kda_backward_tile(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const T* __restrict__ la, int la_scalar, const T* __restrict__ beta,
                  const int32_t* __restrict__ cu, const DeviceHeader* __restrict__ hdr,
                  const int32_t* __restrict__ chunk_first, int H, int64_t T_tot,
                  const float* __restrict__ s0, const T* __restrict__ dout, const float* __restrict__ dfinal,
                  float* __restrict__ ckpt, float* __restrict__ part, float* __restrict__ dv,
                  float* __restrict__ ds0, int only_if_slow) {
    using SM = BwdSmem<D, COLS>;
    constexpr int RP = SM::kRP, RG = SM::kRG;
    constexpr int kTiles = D / COLS;
    if (hdr->status != KDA_OK || (only_if_slow && hdr->pad[kHdrSlowChunk] == 0)) return;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SM& sm = *reinterpret_cast<SM*>(smem_raw);
    const int nh = blockIdx.x, tile = blockIdx.y, n = nh / H, h = nh % H;
    const int col0 = tile * COLS;
    const int tid = threadIdx.x, rg = tid % RG, j = tid / RG, warp = tid >> 5;
    const int64_t t0 = cu[n];
    const int L = (int)(cu[n + 1] - t0);
    // kept states: block b of this sequence at ckpt[((blk0 + b) * H + h) * kTiles + tile]
    const int64_t blk0 = (int64_t)chunk_first[n] * (kChunk / kBlk);
    auto kept = [&](int b) { return ckpt + (((size_t)(blk0 + b) * H + h) * kTiles + tile) * (size_t)D * COLS; };
    const size_t sbase = (size_t)nh * D * D;

    // ---- forward: keep the state at the start of every block
    float S[RP];
#pragma unroll
    for (int a = 0; a < RP; ++a) S[a] = s0 ? s0[sbase + (size_t)(a * RG + rg) * D + col0 + j] : 0.f;
    for (int b = 0; b * kBlk < L; ++b) {
        float* kp = kept(b);
#pragma unroll
        for (int a = 0; a < RP; ++a) kp[(a * COLS + j) * RG + rg] = S[a];
        const int n_b = min(kBlk, L - b * kBlk);
        __syncthreads();
        bwd_load_tokens<T, D, COLS>(sm, t0 + (int64_t)b * kBlk, n_b, h, H, col0, q, k, v, la, la_scalar, beta,
                                    dout);
        __syncthreads();
        for (int r = 0; r < n_b; ++r) bwd_fwd_step<D, COLS>(sm, S, r, rg, j);
    }

    // ---- backward, block by block from the end
    float dS[RP];
#pragma unroll
    for (int a = 0; a < RP; ++a) dS[a] = dfinal ? dfinal[sbase + (size_t)(a * RG + rg) * D + col0 + j] : 0.f;
    const int nblk = (L + kBlk - 1) / kBlk;
    for (int b = nblk - 1; b >= 0; --b) {
        const int n_b = min(kBlk, L - b * kBlk);
        const int64_t tb = t0 + (int64_t)b * kBlk;
        __syncthreads();
        bwd_load_tokens<T, D, COLS>(sm, tb, n_b, h, H, col0, q, k, v, la, la_scalar, beta, dout);
        const float* kp = kept(b);
#pragma unroll
        for (int a = 0; a < RP; ++a) S[a] = kp[(a * COLS + j) * RG + rg];
        __syncthreads();
        // recompute the block: st[r] = S_{t-1} of token r, e[r]
        for (int r = 0; r < n_b; ++r) {
#pragma unroll
            for (int a = 0; a < RP; ++a) sm.st[r][a][j][rg] = S[a];
            const float e = bwd_fwd_step<D, COLS>(sm, S, r, rg, j);
            if (rg == 0) sm.e[r][j] = e;
        }
        __syncthreads();
        for (int r = n_b - 1; r >= 0; --r) {
            float (&red)[3 * D + 1] = sm.red[r & 1][warp];
            const int64_t t = tb + r;
            const float bt = sm.beta[r], e_j = sm.e[r][j], do_j = sm.dout[r][j];
            float Sp[RP], Sprev[RP];
            float pq[RP], pk[RP], pa[RP];
            // read: dq = S_t do, dS += q do^T
            float uk = 0.f;
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const int i = a * RG + rg;
                Sprev[a] = sm.st[r][a][j][rg];
                Sp[a] = sm.alpha[r][i] * Sprev[a];
                const float St = fmaf(sm.k[r][i], bt * e_j, Sp[a]);
                pq[a] = St * do_j;
                dS[a] = fmaf(sm.q[r][i], do_j, dS[a]);
                uk = fmaf(sm.k[r][i], dS[a], uk);
            }
            const float u = rows_sum<RG>(uk);
            const float de = bt * u;
            if (rg == 0) dv[((size_t)t * H + h) * D + col0 + j] = de;
            // write and decay
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const int i = a * RG + rg;
                pk[a] = bt * dS[a] * e_j - Sp[a] * de;
                const float dSp = fmaf(-sm.k[r][i], de, dS[a]);
                pa[a] = dSp * Sprev[a];
                dS[a] = sm.alpha[r][i] * dSp;
            }
            // column sums over the tile of dq, dk, dalpha and dbeta (= e . u):
            // the warp's columns by shuffles, then the 8 warps through red[]
#pragma unroll
            for (int a = 0; a < RP; ++a) {
                const float sq = warp_cols_sum<RG>(pq[a]);
                const float sk = warp_cols_sum<RG>(pk[a]);
                const float sa = warp_cols_sum<RG>(pa[a]);
                if (lane_col0(tid, RG)) {               // row a * RG + rg: consecutive lanes, consecutive words
                    red[a * RG + rg] = sq;
                    red[D + a * RG + rg] = sk;
                    red[2 * D + a * RG + rg] = sa;
                }
            }
            const float eu = warp_cols_sum<RG>(rg == 0 ? e_j * u : 0.f);
            if ((tid & 31) == 0) red[3 * D] = eu;
            __syncthreads();
            float* pt = part + ((size_t)tile * T_tot + t) * H * (3 * D + 1) + (size_t)h * (3 * D + 1);
            for (int w = tid; w <= 3 * D; w += kBwdThreads) {
                const int m = w / D, i = w - m * D;
                float acc = 0.f;
#pragma unroll
                for (int g = 0; g < kBwdThreads / 32; ++g) acc += sm.red[r & 1][g][w];
                pt[w] = m == 2 ? acc * sm.alpha[r][i] : acc;
            }
        }
    }
    if (ds0) {
#pragma unroll
        for (int a = 0; a < RP; ++a) ds0[sbase + (size_t)(a * RG + rg) * D + col0 + j] = dS[a];
    }
}

// Adds the tiles' partial sums: dq, dk, dlog_alpha (per channel, or summed
// over channels for a scalar gate) and dbeta, in tile order.
template <int D>
__global__ void __launch_bounds__(256)
kda_backward_reduce(const float* __restrict__ part, const DeviceHeader* __restrict__ hdr, int64_t T_tot, int H,
                    int kTiles, int la_scalar, float* __restrict__ dq, float* __restrict__ dk,
                    float* __restrict__ dla, float* __restrict__ dbeta, int only_if_slow) {
    constexpr int W = 3 * D + 1;
    if (hdr->status != KDA_OK || (only_if_slow && hdr->pad[kHdrSlowChunk] == 0)) return;
    __shared__ float s_la[D];
    for (int64_t th = blockIdx.x; th < T_tot * H; th += gridDim.x) {   // (token, head)
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
            __syncthreads();
        }
    }
}

size_t backward_ckpt_bytes(int d, int H, int64_t chunks_ub) {
    return (size_t)chunks_ub * (kChunk / kBlk) * H * (size_t)d * d * sizeof(float);
}
// Columns per CTA: fewer when wider tiles would leave SMs idle.
static int bwd_cols(int N, int H, int d) {
    const int64_t nh = (int64_t)N * H;
    return nh * (d / 32) >= 152 ? 32 : nh * (d / 16) >= 152 ? 16 : 8;
}

size_t backward_part_bytes(int N, int d, int H, int64_t T) {
    return (size_t)(d / bwd_cols(N, H, d)) * T * H * (3 * (size_t)d + 1) * sizeof(float);
}

template <typename T, int D, int COLS>
static cudaError_t launch_bwd(const BackwardArgs& a, cudaStream_t stream) {
    cudaError_t e;
    const size_t smem = sizeof(BwdSmem<D, COLS>);
    if ((e = cudaFuncSetAttribute(kda_backward_tile<T, D, COLS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess) return e;
    kda_backward_tile<T, D, COLS><<<dim3((unsigned)a.N * a.H, D / COLS), kBwdThreads, smem, stream>>>(
        (const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.la, a.la_scalar, (const T*)a.beta, a.cu,
        (const DeviceHeader*)a.hdr, a.chunk_first, a.H, a.T, a.s0, (const T*)a.dout, a.dfinal, a.ckpt, a.part,
        a.dv, a.ds0, a.only_if_slow);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.T > 0) {
        const int64_t rows = a.T * a.H;
        kda_backward_reduce<D><<<(unsigned)(rows < 16384 ? rows : 16384), 256, 0, stream>>>(
            a.part, (const DeviceHeader*)a.hdr, a.T, a.H, D / COLS, a.la_scalar, a.dq, a.dk, a.dla, a.dbeta,
            a.only_if_slow);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T, int D>
static cudaError_t launch_bwd_cols(const BackwardArgs& a, cudaStream_t stream) {
    const int cols = bwd_cols(a.N, a.H, D);
    return cols == 8 ? launch_bwd<T, D, 8>(a, stream)
                     : cols == 16 ? launch_bwd<T, D, 16>(a, stream) : launch_bwd<T, D, 32>(a, stream);
}

cudaError_t backward_launch(const BackwardArgs& a, cudaStream_t stream) {
    if (a.dtype == KDA_BF16)
        return a.d == 128 ? launch_bwd_cols<__nv_bfloat16, 128>(a, stream)
                          : launch_bwd_cols<__nv_bfloat16, 64>(a, stream);
    return a.d == 128 ? launch_bwd_cols<float, 128>(a, stream) : launch_bwd_cols<float, 64>(a, stream);
}

}  // namespace kda

// kda_decode.cu -- kernel (c): one recurrent KDA decode step, state updated in place.
//
// Per (sequence, head) the step is ("Kimi Delta Attention" deep dive, section 06,
// fused recurrent KDA; recurrence of section 03, read of section 02):
//
//     S' = Diag(alpha) S            alpha = exp(log_alpha)      [d_k x d_v]
//                                   (one alpha for all rows with the scalar gate)
//     p  = S'^T k                   (what the decayed memory predicts at k)
//     u  = beta (v - p)
//     S  <- S' + k u^T              written back in place
//     o  = S^T q = S'^T q + (k.q) u
//
// Both column reductions p and S'^T q come out of ONE pass over S, so the state
// is read once and written once: the step is bound by HBM bandwidth on the
// 2 * d_k * d_v * 4 bytes of fp32 state per (sequence, head).
//
// Grid: (N*H, d_v / TILE).  A CTA owns a d_k x TILE column tile of one state
// (columns of S are independent); TILE = 64 (97% of the measured copy
// bandwidth on GB300, against 86% with 32-column tiles: fewer, longer CTAs and
// fewer redundant q/k/alpha loads).  256 threads: TILE / 8 threads cover a row
// with 32-byte vectors (the widest global access on sm_100+), 256 / (TILE / 8)
// rows per pass, the passes held in registers between the reduction and the
// update.  State loads are issued before the small q/k/alpha staging so their
// latency overlaps it; loads and stores carry an evict-first L2 hint because
// the state is touched exactly once per step.
#include "kda_common.cuh"
#include "kda_paths.h"

namespace kda {

constexpr int kDecTile = 64;     // state columns per CTA (at most D)
constexpr int kDecThreads = 256;

struct f8 { float v[8]; };

__device__ __forceinline__ f8 ld_stream_f8(const float* p) {
    uint32_t r[8];
    asm volatile("ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
                   "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]) : "l"(p));
    f8 o;
#pragma unroll
    for (int i = 0; i < 8; ++i) o.v[i] = __uint_as_float(r[i]);
    return o;
}
__device__ __forceinline__ void st_stream_f8(float* p, const f8& x) {
    asm volatile("st.global.L1::no_allocate.L2::evict_first.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(__float_as_uint(x.v[0])), "r"(__float_as_uint(x.v[1])),
                    "r"(__float_as_uint(x.v[2])), "r"(__float_as_uint(x.v[3])),
                    "r"(__float_as_uint(x.v[4])), "r"(__float_as_uint(x.v[5])),
                    "r"(__float_as_uint(x.v[6])), "r"(__float_as_uint(x.v[7])) : "memory");
}

template <typename T, int D, int TILE>
__global__ void __launch_bounds__(kDecThreads)
kda_decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const T* __restrict__ log_alpha, int la_scalar, const T* __restrict__ beta,
                       float* __restrict__ state, T* __restrict__ out, int H) {
    constexpr int kTPR = TILE / 8;                  // threads per row of the tile (8 floats each)
    constexpr int kRowsPerPass = kDecThreads / kTPR;
    constexpr int kPasses = D / kRowsPerPass;       // rows per thread
    const int nh = blockIdx.x;                      // (sequence, head) pair, = n * H + h
    const int col0 = blockIdx.y * TILE;
    const int tid = threadIdx.x;
    const int rsub = tid / kTPR;                    // row within a pass
    const int c8 = tid % kTPR;                      // which 8-float group of the tile

    float* S = state + (size_t)nh * D * D;
    f8 s[kPasses];
#pragma unroll
    for (int p = 0; p < kPasses; ++p)
        s[p] = ld_stream_f8(S + (size_t)(p * kRowsPerPass + rsub) * D + col0 + c8 * 8);

    __shared__ float sh_alpha[D], sh_k[D], sh_q[D];
    __shared__ float sh_red[kDecThreads / 32][2][TILE];
    __shared__ __align__(16) float sh_u[TILE];
    __shared__ float sh_kq;

    const size_t vec = (size_t)nh * D;              // q, k, log_alpha, v rows of this (n, h)
    if (tid < D) {
        sh_alpha[tid] = expf(to_f32(log_alpha[la_scalar ? (size_t)nh : vec + tid]));
        sh_k[tid] = to_f32(k[vec + tid]);
        sh_q[tid] = to_f32(q[vec + tid]);
    }
    __syncthreads();
    if (tid < 32) {                                 // k . q over the full key dimension
        float a = 0.f;
        for (int i = tid; i < D; i += 32) a += sh_k[i] * sh_q[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (tid == 0) sh_kq = a;
    }

    // Partial column sums of S'^T k and S'^T q over this thread's rows.
    float pk[8], pq[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { pk[j] = 0.f; pq[j] = 0.f; }
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
        const int r = p * kRowsPerPass + rsub;
        const float a = sh_alpha[r], kr = sh_k[r], qr = sh_q[r];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s[p].v[j] *= a;                         // S' = Diag(alpha) S
            pk[j] += kr * s[p].v[j];
            pq[j] += qr * s[p].v[j];
        }
    }
    // Reduce over the row groups of a warp (lanes kTPR, 2 kTPR, ... apart).
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int o = kTPR; o < 32; o <<= 1) {
            pk[j] += __shfl_xor_sync(0xffffffffu, pk[j], o);
            pq[j] += __shfl_xor_sync(0xffffffffu, pq[j], o);
        }
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < kTPR) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sh_red[warp][0][lane * 8 + j] = pk[j];
            sh_red[warp][1][lane * 8 + j] = pq[j];
        }
    }
    __syncthreads();
    if (tid < TILE) {
        float p = 0.f, r = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) { p += sh_red[w][0][tid]; r += sh_red[w][1][tid]; }
        const int j = col0 + tid;
        const float b = to_f32(beta[nh]);
        const float u = b * (to_f32(v[vec + j]) - p);   // u = beta (v - S'^T k)
        sh_u[tid] = u;
        out[vec + j] = from_f32<T>(r + sh_kq * u);      // o = S'^T q + (k.q) u
    }
    __syncthreads();
    float u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) u[j] = sh_u[c8 * 8 + j];
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
        const int r = p * kRowsPerPass + rsub;
        const float kr = sh_k[r];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[p].v[j] += kr * u[j];   // S' + k u^T
        st_stream_f8(S + (size_t)r * D + col0 + c8 * 8, s[p]);
    }
}

template <typename T, int D>
static cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* la,
                                 int la_scalar, const void* beta, float* state, void* out, int N, int H,
                                 cudaStream_t stream) {
    constexpr int kTile = kDecTile < D ? kDecTile : D;
    dim3 grid((unsigned)N * H, D / kTile);
    kda_decode_step_kernel<T, D, kTile><<<grid, kDecThreads, 0, stream>>>(
        (const T*)q, (const T*)k, (const T*)v, (const T*)la, la_scalar, (const T*)beta, state, (T*)out, H);
    return cudaGetLastError();
}

cudaError_t decode_step_launch(int dtype, int d, const void* q, const void* k, const void* v,
                               const void* la, int la_scalar, const void* beta, float* state, void* out,
                               int N, int H, cudaStream_t stream) {
    if (dtype == KDA_BF16)
        return d == 128 ? launch_decode<__nv_bfloat16, 128>(q, k, v, la, la_scalar, beta, state, out, N, H, stream)
                        : launch_decode<__nv_bfloat16, 64>(q, k, v, la, la_scalar, beta, state, out, N, H, stream);
    return d == 128 ? launch_decode<float, 128>(q, k, v, la, la_scalar, beta, state, out, N, H, stream)
                    : launch_decode<float, 64>(q, k, v, la, la_scalar, beta, state, out, N, H, stream);
}

}  // namespace kda

// kda_api.cu -- the C ABI declared in include/kda.h: argument checks, the
// workspace layout, the sequence-table kernel and the dispatch to kernels.
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_paths.h"

namespace kda {

static thread_local int g_last_cuda_error = 0;

static int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return KDA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Sequence table: checks cu_seqlens and turns it into per-sequence chunk
// offsets (exclusive prefix of ceil(len / kChunk)).  One CTA; no host sync.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads)
kda_sequence_table(const int32_t* __restrict__ cu_in, int N, int64_t T_tot, DeviceHeader* hdr,
                   int32_t* __restrict__ chunk_first, int64_t chunks_ub) {
    __shared__ int s_bad;
    __shared__ long long s_carry;
    __shared__ long long s_warp[kPrepThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* cu_local = hdr->pad;               // used when the caller passes no cu_seqlens
    const int32_t* cu = cu_in;
    if (cu_in == nullptr) {
        if (tid == 0) { cu_local[0] = 0; cu_local[1] = (int32_t)T_tot; }
        __syncthreads();
        cu = cu_local;
    }
    if (tid == 0) {
        s_bad = (cu[0] != 0 || (int64_t)cu[N] != T_tot) ? 1 : 0;
        s_carry = 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += kPrepThreads) {
        const int i = base + tid;
        long long cnt = 0;
        if (i < N) {
            const int32_t a = cu[i], b = cu[i + 1];
            if (b < a) s_bad = 1;
            else cnt = ((long long)b - a + kChunk - 1) / kChunk;
        }
        long long x = cnt;                       // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            long long w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                long long y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_warp[lane] = w;                    // inclusive over warps
        }
        __syncthreads();
        const long long excl = s_carry + (warp ? s_warp[warp - 1] : 0) + x - cnt;
        if (i < N) chunk_first[i] = (int32_t)min64(excl, 0x7fffffffLL);
        __syncthreads();
        if (tid == 0) s_carry += s_warp[kPrepThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) {
        const long long total = s_carry;
        const int bad = s_bad || total > chunks_ub;
        chunk_first[N] = (int32_t)min64(total, 0x7fffffffLL);
        hdr->total_chunks = bad ? 0 : (int32_t)total;
        hdr->pad[kHdrSlowChunk] = 0;
        hdr->status = bad ? KDA_ERR_BAD_SEQLENS : KDA_OK;
    }
}

// ---------------------------------------------------------------------------
// Snapshot requests: one CTA per request (sequence n, prefix length p).  A
// request at p = 0 copies the initial state; any other marks the chunk that
// ends at p, whose state the inter-chunk kernels write out after processing
// it.  Checks every request; a bad or repeated one sets KDA_ERR_BAD_SNAPSHOT.
// slot[] holds -1 on entry (set by the caller's memset).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
kda_snapshot_table(const int32_t* __restrict__ at, const int32_t* __restrict__ cu, const int32_t* chunk_first,
                   int N, int H, int D, DeviceHeader* hdr, int32_t* slot, const float* __restrict__ s0,
                   float* __restrict__ snaps) {
    if (hdr->status != KDA_OK) return;
    const int m = blockIdx.x;
    const int n = at[2 * m], p = at[2 * m + 1];
    if (n < 0 || n >= N) { if (threadIdx.x == 0) record_status(hdr, KDA_ERR_BAD_SNAPSHOT); return; }
    const int len = cu[n + 1] - cu[n];
    if (p < 0 || p > len || (p % kChunk != 0 && p != len)) {
        if (threadIdx.x == 0) record_status(hdr, KDA_ERR_BAD_SNAPSHOT);
        return;
    }
    if (p == 0) {                                  // the state before any token
        const size_t per = (size_t)H * D * D;
        float4* dst = (float4*)(snaps + (size_t)m * per);
        const float4* src = s0 ? (const float4*)(s0 + (size_t)n * per) : nullptr;
        for (size_t e = threadIdx.x; e < per / 4; e += blockDim.x)
            dst[e] = src ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (threadIdx.x == 0) {
        const int c = chunk_first[n] + (p + kChunk - 1) / kChunk - 1;
        if (atomicCAS(&slot[c], -1, m) != -1) record_status(hdr, KDA_ERR_BAD_SNAPSHOT);
    }
}

// ---------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    int path;              // which prefill path runs
    int64_t chunks_ub;     // upper bound on total chunks: ceil(T/C) + N
    size_t table_off;      // int32 chunk_first[N+1]
    size_t slot_off;       // int32 snapshot slot per chunk [chunks_ub]
    size_t rec_off;        // per-(chunk, head) records
    size_t rec_bytes;
    size_t extra_off;      // path-specific scratch
    size_t total;
};

static Layout layout_for(const kda_desc* d) {
    Layout L;
    L.path = choose_prefill_path(d->dtype, d->d_k, d->flags);
    L.chunks_ub = (d->total_tokens + kChunk - 1) / kChunk + d->num_seqs;
    L.table_off = sizeof(DeviceHeader);
    L.slot_off = align_up(L.table_off + ((size_t)d->num_seqs + 1) * sizeof(int32_t), 256);
    L.rec_off = align_up(L.slot_off + (size_t)L.chunks_ub * sizeof(int32_t), 1024);
    L.rec_bytes = prefill_record_bytes(L.path, d->d_k);
    L.extra_off = align_up(L.rec_off + (size_t)L.chunks_ub * d->num_heads * L.rec_bytes, 1024);
    L.total = L.extra_off + prefill_extra_bytes(L.path, d->num_seqs, d->num_heads, d->total_tokens);
    return L;
}

static bool desc_ok(const kda_desc* d) {
    if (!d) return false;
    if (d->num_seqs < 0 || d->num_heads < 1 || d->total_tokens < 0) return false;
    if (d->flags & ~(KDA_FLAG_CUDA_CORE_PREFILL | KDA_FLAG_SCALAR_GATE)) return false;
    if (d->total_tokens > 0x7fffffffLL) return false;   // cu_seqlens is int32
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return false;
    if (d->d_k < 1 || d->d_v < 1) return false;
    return true;
}

static bool shape_supported(const kda_desc* d) {
    return d->d_k == d->d_v && (d->d_k == 64 || d->d_k == 128);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace kda

using namespace kda;

extern "C" {

int kda_version(void) { return 10000; }

int kda_last_cuda_error(void) { return g_last_cuda_error; }

const char* kda_status_string(int s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_BAD_SEQLENS: return "KDA_ERR_BAD_SEQLENS";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_BAD_SNAPSHOT: return "KDA_ERR_BAD_SNAPSHOT";
        default: return "KDA_ERR_UNKNOWN";
    }
}

size_t kda_prefill_workspace_bytes(const kda_desc* d) {
    if (!desc_ok(d) || !shape_supported(d)) return 0;
    return layout_for(d).total;
}

static int prefill_impl(const kda_desc* d, const void* q, const void* k, const void* v,
                        const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                        const float* initial_state, void* out, float* final_state, int32_t num_snaps,
                        const int32_t* snap_at, float* snaps, kda_stream_t stream) {
    if (!desc_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
    if (!shape_supported(d)) return KDA_ERR_UNSUPPORTED;
    const int N = d->num_seqs, H = d->num_heads, D = d->d_k;
    const int64_t T = d->total_tokens;
    if (cu_seqlens == nullptr && N != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    const size_t esz = d->dtype == KDA_BF16 ? 2 : 4;
    const bool scalar_gate = (d->flags & KDA_FLAG_SCALAR_GATE) != 0;
    const size_t nqk = (size_t)T * H * D * esz, nb = (size_t)T * H * esz;
    const size_t nla = scalar_gate ? nb : nqk;
    const size_t nstate = (size_t)N * H * D * D * sizeof(float);
    if (T > 0) {
        if (!q || !k || !v || !log_alpha || !beta || !out) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
            (scalar_gate ? ((uintptr_t)log_alpha % esz) != 0 : !aligned16(log_alpha)) ||
            ((uintptr_t)beta % esz) || !aligned16(out)) return KDA_ERR_INVALID_ARGUMENT;
        const void* ins[5] = {q, k, v, log_alpha, beta};
        const size_t szs[5] = {nqk, nqk, nqk, nla, nb};
        for (int i = 0; i < 5; ++i)
            if (overlaps(out, nqk, ins[i], szs[i])) return KDA_ERR_INVALID_ARGUMENT;
        if (overlaps(out, nqk, initial_state, nstate) || overlaps(out, nqk, final_state, nstate))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((cu_seqlens && !aligned16(cu_seqlens)) || (initial_state && !aligned16(initial_state)) ||
        (final_state && !aligned16(final_state))) return KDA_ERR_INVALID_ARGUMENT;
    if (initial_state && final_state && initial_state != (const float*)final_state &&
        overlaps(initial_state, nstate, final_state, nstate)) return KDA_ERR_INVALID_ARGUMENT;
    if (num_snaps < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (num_snaps > 0) {
        if (!snap_at || !snaps || ((uintptr_t)snap_at & 3u) || !aligned16(snaps)) return KDA_ERR_INVALID_ARGUMENT;
        const size_t nsnap = (size_t)num_snaps * H * D * D * sizeof(float);
        const size_t nat = (size_t)num_snaps * 2 * sizeof(int32_t);
        const void* bufs[9] = {q, k, v, log_alpha, beta, out, initial_state, final_state, snap_at};
        const size_t szs[9] = {nqk, nqk, nqk, nla, nb, nqk, nstate, nstate, nat};
        for (int i = 0; i < 9; ++i)
            if (overlaps(snaps, nsnap, bufs[i], szs[i])) return KDA_ERR_INVALID_ARGUMENT;
    }
    const Layout L = layout_for(d);
    if (!d->workspace || d->workspace_bytes < L.total || ((uintptr_t)d->workspace & 255u))
        return KDA_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d->workspace;
    DeviceHeader* hdr = (DeviceHeader*)ws;
    int32_t* chunk_first = (int32_t*)(ws + L.table_off);
    kda_sequence_table<<<1, kPrepThreads, 0, s>>>(cu_seqlens, N, T, hdr, chunk_first, L.chunks_ub);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    int32_t* slot = (int32_t*)(ws + L.slot_off);
    if (num_snaps > 0) {
        if ((e = cudaMemsetAsync(slot, 0xff, (size_t)L.chunks_ub * sizeof(int32_t), s)) != cudaSuccess)
            return cuda_fail(e);
        kda_snapshot_table<<<num_snaps, 256, 0, s>>>(snap_at, cu_seqlens ? cu_seqlens : hdr->pad, chunk_first, N, H,
                                                     D, hdr, slot, initial_state, snaps);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    }
    PrefillArgs a;
    a.dtype = d->dtype; a.d = D; a.N = N; a.H = H; a.chunks_ub = (int)L.chunks_ub; a.T = T;
    a.q = q; a.k = k; a.v = v; a.la = log_alpha; a.beta = beta; a.la_scalar = scalar_gate ? 1 : 0;
    a.cu = cu_seqlens ? cu_seqlens : hdr->pad;
    a.s0 = initial_state; a.out = out; a.sf = final_state;
    a.hdr = hdr; a.chunk_first = chunk_first; a.recs = ws + L.rec_off; a.extra = ws + L.extra_off;
    a.phase_events = (cudaEvent_t*)d->phase_events;
    a.snap_slot = num_snaps > 0 ? slot : nullptr;
    a.snaps = num_snaps > 0 ? snaps : nullptr;
    e = prefill_launch(L.path, a, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return KDA_OK;
}

int kda_prefill(const kda_desc* d, const void* q, const void* k, const void* v,
                const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                const float* initial_state, void* out, float* final_state, kda_stream_t stream) {
    return prefill_impl(d, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state, 0, nullptr,
                             nullptr, stream);
}

int kda_prefill_snapshots(const kda_desc* d, const void* q, const void* k, const void* v,
                          const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                          const float* initial_state, void* out, float* final_state, int32_t num_snapshots,
                          const int32_t* snapshot_at, float* snapshots, kda_stream_t stream) {
    return prefill_impl(d, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                             num_snapshots, snapshot_at, snapshots, stream);
}

// Backward workspace: header, chunk table, then the CUDA-core backward's kept
// states and per-tile partial sums.  On the tensor-core path the same region
// (from ckpt_off) first holds the tensor-core backward's scratch; the
// CUDA-core kernels run after it only as its fallback, when the tensor-core
// kernels have returned without work, so the two uses may overlap.
struct BwdLayout {
    bool tc;               // tensor-core backward (bf16, head size 128)
    int64_t chunks_ub;
    size_t table_off, ckpt_off, part_off, total;
};
static bool bwd_uses_tc(const kda_desc* d) {
    return d->dtype == KDA_BF16 && d->d_k == 128 && (d->flags & KDA_FLAG_CUDA_CORE_PREFILL) == 0;
}
static BwdLayout bwd_layout(const kda_desc* d) {
    BwdLayout L;
    L.tc = bwd_uses_tc(d);
    L.chunks_ub = (d->total_tokens + kChunk - 1) / kChunk + d->num_seqs;
    L.table_off = sizeof(DeviceHeader);
    L.ckpt_off = align_up(L.table_off + ((size_t)d->num_seqs + 1) * sizeof(int32_t), 1024);
    L.part_off = align_up(L.ckpt_off + backward_ckpt_bytes(d->d_k, d->num_heads, L.chunks_ub), 1024);
    L.total = L.part_off + backward_part_bytes(d->num_seqs, d->d_k, d->num_heads, d->total_tokens);
    if (L.tc) {
        const size_t tc_end = L.ckpt_off + backward_tc_bytes(d->num_seqs, d->num_heads, d->total_tokens, L.chunks_ub);
        if (tc_end > L.total) L.total = tc_end;
    }
    return L;
}

size_t kda_backward_workspace_bytes(const kda_desc* d) {
    if (!desc_ok(d) || !shape_supported(d)) return 0;
    return bwd_layout(d).total;
}

int kda_prefill_backward(const kda_desc* d, const void* q, const void* k, const void* v,
                         const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                         const float* initial_state, const void* d_out, const float* d_final_state, float* dq,
                         float* dk, float* dv, float* dlog_alpha, float* dbeta, float* d_initial_state,
                         kda_stream_t stream) {
    if (!desc_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
    if (!shape_supported(d)) return KDA_ERR_UNSUPPORTED;
    const int N = d->num_seqs, H = d->num_heads, D = d->d_k;
    const int64_t T = d->total_tokens;
    if (cu_seqlens == nullptr && N != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    const size_t esz = d->dtype == KDA_BF16 ? 2 : 4;
    const bool scalar_gate = (d->flags & KDA_FLAG_SCALAR_GATE) != 0;
    const size_t nqk = (size_t)T * H * D * esz, nb = (size_t)T * H * esz, nla = scalar_gate ? nb : nqk;
    const size_t g_qk = (size_t)T * H * D * 4, g_b = (size_t)T * H * 4, g_la = scalar_gate ? g_b : g_qk;
    const size_t nstate = (size_t)N * H * D * D * sizeof(float);
    if (T > 0) {
        if (!q || !k || !v || !log_alpha || !beta || !d_out || !dq || !dk || !dv || !dlog_alpha || !dbeta)
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(d_out) ||
            (scalar_gate ? ((uintptr_t)log_alpha % esz) != 0 : !aligned16(log_alpha)) || ((uintptr_t)beta % esz))
            return KDA_ERR_INVALID_ARGUMENT;
        if (((uintptr_t)dq | (uintptr_t)dk | (uintptr_t)dv | (uintptr_t)dlog_alpha | (uintptr_t)dbeta) & 3u)
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((cu_seqlens && !aligned16(cu_seqlens)) || (initial_state && !aligned16(initial_state)) ||
        (d_final_state && !aligned16(d_final_state)) || (d_initial_state && !aligned16(d_initial_state)))
        return KDA_ERR_INVALID_ARGUMENT;
    // outputs may not overlap inputs or one another
    const void* outs[6] = {dq, dk, dv, dlog_alpha, dbeta, d_initial_state};
    const size_t osz[6] = {g_qk, g_qk, g_qk, g_la, g_b, nstate};
    const void* ins[9] = {q, k, v, log_alpha, beta, d_out, initial_state, d_final_state, cu_seqlens};
    const size_t isz[9] = {nqk, nqk, nqk, nla, nb, nqk, nstate, nstate, ((size_t)N + 1) * 4};
    for (int a = 0; a < 6; ++a) {
        for (int b = 0; b < 9; ++b)
            if (overlaps(outs[a], osz[a], ins[b], isz[b])) return KDA_ERR_INVALID_ARGUMENT;
        for (int b = a + 1; b < 6; ++b)
            if (overlaps(outs[a], osz[a], outs[b], osz[b])) return KDA_ERR_INVALID_ARGUMENT;
    }
    const BwdLayout L = bwd_layout(d);
    if (!d->workspace || d->workspace_bytes < L.total || ((uintptr_t)d->workspace & 255u)) return KDA_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d->workspace;
    DeviceHeader* hdr = (DeviceHeader*)ws;
    int32_t* chunk_first = (int32_t*)(ws + L.table_off);
    kda_sequence_table<<<1, kPrepThreads, 0, s>>>(cu_seqlens, N, T, hdr, chunk_first, L.chunks_ub);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    BackwardArgs a;
    a.dtype = d->dtype; a.d = D; a.N = N; a.H = H; a.T = T;
    a.q = q; a.k = k; a.v = v; a.la = log_alpha; a.beta = beta; a.dout = d_out; a.la_scalar = scalar_gate ? 1 : 0;
    a.cu = cu_seqlens ? cu_seqlens : hdr->pad;
    a.s0 = initial_state; a.dfinal = d_final_state;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dla = dlog_alpha; a.dbeta = dbeta; a.ds0 = d_initial_state;
    a.hdr = hdr; a.chunk_first = chunk_first;
    a.ckpt = (float*)(ws + L.ckpt_off); a.part = (float*)(ws + L.part_off);
    a.only_if_slow = 0;
    if (L.tc) {
        if ((e = backward_tc_launch(a, L.chunks_ub, ws + L.ckpt_off, s)) != cudaSuccess) return cuda_fail(e);
        a.only_if_slow = 1;         // the CUDA-core kernels below return unless a chunk was too strong
    }
    if ((e = backward_launch(a, s)) != cudaSuccess) return cuda_fail(e);
    return KDA_OK;
}

int kda_decode_step(const kda_desc* d, const void* q, const void* k, const void* v,
                    const void* log_alpha, const void* beta, float* state_inout, void* out,
                    kda_stream_t stream) {
    if (!desc_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
    if (!shape_supported(d)) return KDA_ERR_UNSUPPORTED;
    const int N = d->num_seqs, H = d->num_heads, D = d->d_k;
    if (d->total_tokens != N) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !state_inout || !out) return KDA_ERR_INVALID_ARGUMENT;
    const size_t esz = d->dtype == KDA_BF16 ? 2 : 4;
    const bool scalar_gate = (d->flags & KDA_FLAG_SCALAR_GATE) != 0;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
        (scalar_gate ? ((uintptr_t)log_alpha % esz) != 0 : !aligned16(log_alpha)) || ((uintptr_t)beta % esz) ||
        ((uintptr_t)state_inout & 31u) || !aligned16(out)) return KDA_ERR_INVALID_ARGUMENT;
    if ((int64_t)N * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARGUMENT;
    const size_t nio = (size_t)N * H * D * esz, nstate = (size_t)N * H * D * D * sizeof(float);
    const size_t nsc = (size_t)N * H * esz;
    const void* ins[5] = {q, k, v, log_alpha, beta};
    const size_t szs[5] = {nio, nio, nio, scalar_gate ? nsc : nio, nsc};
    for (int i = 0; i < 5; ++i)
        if (overlaps(out, nio, ins[i], szs[i]) || overlaps(state_inout, nstate, ins[i], szs[i]))
            return KDA_ERR_INVALID_ARGUMENT;
    if (overlaps(out, nio, state_inout, nstate)) return KDA_ERR_INVALID_ARGUMENT;
    cudaError_t e = decode_step_launch(d->dtype, D, q, k, v, log_alpha, scalar_gate ? 1 : 0, beta, state_inout,
                                       out, N, H, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return KDA_OK;
}

int kda_get_device_status(const kda_desc* d, kda_stream_t stream) {
    if (!d || !d->workspace || d->workspace_bytes < sizeof(DeviceHeader)) return KDA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t status = 0;
    cudaError_t e = cudaMemcpyAsync(&status, d->workspace, sizeof(status), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return status;
}

}  // extern "C"

namespace kda {

int choose_prefill_path(int dtype, int d, int flags) {
    if ((flags & KDA_FLAG_CUDA_CORE_PREFILL) == 0 && dtype == KDA_BF16 && d == 128) return kPathTensorCore;
    return kPathSimt;
}

size_t prefill_record_bytes(int path, int d) {
    return path == kPathTensorCore ? tc_record_bytes() : simt_record_bytes(d);
}

size_t prefill_extra_bytes(int path, int N, int H, int64_t T) {
    return path == kPathTensorCore ? tc_extra_bytes(N, H, T) : 0;
}

cudaError_t prefill_launch(int path, const PrefillArgs& a, cudaStream_t stream) {
    if (path == kPathTensorCore) return prefill_tc_launch(a, a.T, stream);
    return prefill_simt_launch(a, stream);
}

}  // namespace kda

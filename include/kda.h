/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention hot path.
 *
 * The operator (page "Kimi Delta Attention" deep dive, section 03, the
 * recurrence as written in the Kimi Linear report; section 02 for the read):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * per sequence and head, with a fixed d_k x d_v state S (rows are key
 * channels), alpha_t in (0,1]^{d_k} a per-channel decay and beta_t a scalar.
 * It runs in the two modes of section 06 of the same page: a chunk-parallel
 * prefill over a packed batch of variable-length sequences, and a one-token
 * recurrent decode step that updates the state in place.  Section 07 gives the
 * state hand-off: the final state of a prefill is the checkpoint another
 * prefill or the decode step continues from.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every pointer argument is a DEVICE pointer (CUDA global memory of the
 *    current device), row-major and densely packed.  Alignment: q, k, v,
 *    log_alpha, out, cu_seqlens and the prefill states 16 bytes; the decode
 *    state 32 bytes; beta its element size; the workspace 256 bytes.
 *  - Layouts: q, k, log_alpha [T_tot, H, d_k]; v, out [T_tot, H, d_v];
 *    beta [T_tot, H]; cu_seqlens int32 [N+1]; states fp32 [N, H, d_k, d_v]
 *    (d_v contiguous).  The decode step uses the same layouts with T_tot = N.
 *    With KDA_FLAG_SCALAR_GATE, log_alpha is [T_tot, H] instead.
 *  - dtype (KDA_F32 or KDA_BF16) applies to q, k, v, log_alpha, beta and out;
 *    states are always fp32; all accumulation is fp32.
 *  - alpha = exp(log_alpha) is formed inside the kernels; beta is taken as
 *    given (already through its sigmoid).  Scaling and normalising q and k is
 *    the caller's business.
 *  - Supported head sizes: d_k == d_v, 64 or 128 (else KDA_ERR_UNSUPPORTED).
 *  - The caller owns all memory.  The library never allocates or frees
 *    device memory and never synchronises, except kda_get_device_status,
 *    which synchronises the stream it is given.  Work is enqueued on
 *    `stream` (NULL = the legacy default stream); buffers must stay alive
 *    until that work completes.  Calls are re-entrant; concurrent calls on
 *    different streams need different workspaces.
 *  - Return codes are synchronous and report what the host can see (bad
 *    arguments, launch failures).  Problems only the device can detect
 *    (a malformed cu_seqlens) are written to a status word inside the
 *    workspace and read back with kda_get_device_status.  Nothing is thrown
 *    across the ABI.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* null / misaligned pointer, bad size, aliasing out with an input */
    KDA_ERR_UNSUPPORTED = 2,      /* head size or dtype outside what the kernels implement */
    KDA_ERR_CUDA = 3,             /* a CUDA launch or API call failed (see kda_last_cuda_error) */
    KDA_ERR_TIMEOUT = 4,          /* a bounded on-device wait gave up (device status only) */
    KDA_ERR_BAD_SEQLENS = 5,      /* cu_seqlens not 0 = c_0 <= c_1 <= ... <= c_N = T_tot (device status) */
    KDA_ERR_WORKSPACE = 6,        /* workspace missing or smaller than kda_prefill_workspace_bytes */
    KDA_ERR_BAD_SNAPSHOT = 7      /* a snapshot request off its sequence, off a chunk boundary, or
                                     repeated (device status, kda_prefill_snapshots) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* kda_desc.flags bits. */
enum {
    /* Run the prefill (and kda_prefill_backward) on CUDA cores in fp32 even
       where the tensor-core path applies (bf16, head size 128).  Slower; meant
       for cross-checking. */
    KDA_FLAG_CUDA_CORE_PREFILL = 1,
    /* Scalar gate: log_alpha holds ONE value per (token, head) -- layout
       [T_tot, H] for the prefill, [N, H] for the decode step, aligned to its
       element size like beta -- and every key channel of the head decays by
       that same alpha.  This is the Gated DeltaNet gate that KDA refines into
       a per-channel one (deep dive, section 03: Gated DeltaNet multiplies a
       head's state by a scalar alpha, KDA by Diag(alpha)); the result equals
       the per-channel operator with log_alpha broadcast over d_k. */
    KDA_FLAG_SCALAR_GATE = 2
};

/* Problem description.  Not retained by the library after a call returns. */
typedef struct kda_desc {
    int32_t num_seqs;       /* N >= 0 sequences (decode: sequences advanced by one token) */
    int32_t num_heads;      /* H >= 1 */
    int32_t d_k;            /* key/query head size: 64 or 128 */
    int32_t d_v;            /* value head size: must equal d_k */
    int64_t total_tokens;   /* T_tot = cu_seqlens[N] (decode: must equal N) */
    int32_t dtype;          /* kda_dtype of q, k, v, log_alpha, beta, out */
    int32_t flags;          /* OR of KDA_FLAG_* bits (0: tensor cores where they apply, per-channel gate) */
    void *workspace;        /* device scratch owned by the caller (prefill only), 256-byte aligned */
    size_t workspace_bytes; /* its size in bytes */
    void **phase_events;    /* optional timing hook (NULL: none): kda_prefill records
                               phase_events[0] before the intra-chunk kernel,
                               phase_events[1] between it and the inter-chunk kernel and
                               phase_events[2] after that, each a cudaEvent_t created by
                               the caller, on `stream` */
} kda_desc;

/*
 * Bytes of device workspace kda_prefill needs for this description (0 for an
 * invalid one).  The bound depends only on N, H, d and T_tot, never on the
 * contents of cu_seqlens, so it can be sized before the lengths are known on
 * the host.  The workspace is scratch: its contents on entry are ignored, and
 * on exit it holds intermediate chunk data plus the device status word.
 */
KDA_API size_t kda_prefill_workspace_bytes(const kda_desc *desc);

/*
 * Chunk-parallel prefill over a packed batch (deep dive section 06, "chunk-
 * parallel KDA"; variable-length batching per the FlashKDA update there).
 *
 *   q, k, log_alpha  [T_tot, H, d_k]   inputs, dtype `desc->dtype`
 *                    (log_alpha [T_tot, H] with KDA_FLAG_SCALAR_GATE)
 *   v                [T_tot, H, d_v]
 *   beta             [T_tot, H]
 *   cu_seqlens       int32 [N+1], device; sequence n is packed tokens
 *                    [cu_seqlens[n], cu_seqlens[n+1]).  NULL means one
 *                    sequence of all T_tot tokens (then N must be 1).
 *   initial_state    fp32 [N, H, d_k, d_v] or NULL (zero state).
 *   out              [T_tot, H, d_v], written; must not overlap any input.
 *   final_state      fp32 [N, H, d_k, d_v] or NULL (not written).  May be the
 *                    same pointer as initial_state (in-place continuation).
 *                    A sequence of length 0 returns its initial state.
 *   stream           CUDA stream for all work.
 *
 * Returns KDA_OK once the work is enqueued.  A malformed cu_seqlens is not
 * seen by the host: the kernels then skip all work, leave out/final_state
 * unspecified and record KDA_ERR_BAD_SEQLENS in the device status word.
 */
KDA_API int kda_prefill(const kda_desc *desc,
                const void *q, const void *k, const void *v,
                const void *log_alpha, const void *beta,
                const int32_t *cu_seqlens, const float *initial_state,
                void *out, float *final_state, kda_stream_t stream);

/*
 * kda_prefill that also saves the recurrent state at interior positions: the
 * prefix checkpoints of deep dive section 07 (a cached prefix is the state
 * after it; restoring that state and feeding the rest of the sequence
 * continues exactly), taken in the same pass instead of one call per prefix.
 *
 *   num_snapshots  M >= 0 requests.
 *   snapshot_at    int32 [M][2], device, 4-byte aligned: (sequence n, prefix
 *                  length p) pairs, 0 <= n < N, 0 <= p <= L_n, where p is a
 *                  multiple of 64 (the prefill's chunk size) or p = L_n.
 *                  p = 0 gives the initial state.  No pair may repeat.
 *   snapshots      fp32 [M, H, d_k, d_v], device, 16-byte aligned, written:
 *                  snapshot m is the state of sequence n after its first p
 *                  tokens (what kda_prefill over those tokens would return as
 *                  final_state).  Must not overlap any other buffer.
 *
 * Every other argument is that of kda_prefill.  A request that breaks the
 * rules above is seen on the device only: all work is skipped and the status
 * word holds KDA_ERR_BAD_SNAPSHOT.  M = 0 is plain kda_prefill.
 */
KDA_API int kda_prefill_snapshots(const kda_desc *desc,
                                  const void *q, const void *k, const void *v,
                                  const void *log_alpha, const void *beta,
                                  const int32_t *cu_seqlens, const float *initial_state,
                                  void *out, float *final_state,
                                  int32_t num_snapshots, const int32_t *snapshot_at, float *snapshots,
                                  kda_stream_t stream);

/*
 * Reverse mode of kda_prefill: the gradients of a scalar loss with respect to
 * every input, given its gradients with respect to the outputs and the final
 * state.  The deep dive (section 06) names prefill and training as the uses
 * of the chunked form; this entry point supplies the training half by the
 * chain rule through each token's step of the section 03 recurrence.
 *
 *   q, k, v, log_alpha, beta, cu_seqlens, initial_state: as for kda_prefill
 *                    (the same call's inputs).
 *   d_out            [T_tot, H, d_v], dtype `desc->dtype`: dLoss/dout.
 *   d_final_state    fp32 [N, H, d_k, d_v] or NULL (zero): dLoss/dfinal_state.
 *   dq, dk           fp32 [T_tot, H, d_k], written.
 *   dv               fp32 [T_tot, H, d_v], written.
 *   dlog_alpha       fp32 [T_tot, H, d_k] ([T_tot, H] with the scalar gate).
 *   dbeta            fp32 [T_tot, H].
 *   d_initial_state  fp32 [N, H, d_k, d_v] or NULL (not written).
 * Gradients are 4-byte aligned, the states 16-byte aligned; no output may
 * overlap an input or another output.  desc->workspace must hold
 * kda_backward_workspace_bytes(desc) bytes (about 4 * H * d_k * d_v bytes
 * per 8 tokens of kept states plus 4 * (3 d_k + 1) * H * d_v / 32 bytes per
 * token of partial sums, which also covers the tensor-core path's scratch).
 *
 * bf16 inputs with head size 128 run on the tensor cores: the forward is
 * recomputed saving every 64-token chunk's end state, a reverse walk over the
 * chunks gives each chunk's end-state gradient, and one kernel per (chunk,
 * head) forms the gradients (bf16 operands, fp32 accumulation: gradients
 * within about 1e-2 relative L2 of exact arithmetic).  A call in which some
 * chunk's cumulative decay exceeds 2^100 in a channel (log alpha summed over
 * the chunk below -69) runs instead on the fp32 CUDA-core path, decided on
 * the device.  fp32 inputs, head size 64, or KDA_FLAG_CUDA_CORE_PREFILL take
 * the fp32 CUDA-core path (about 1e-4).  Results do not depend on scheduling
 * (no atomics).  Errors as for kda_prefill.
 */
KDA_API size_t kda_backward_workspace_bytes(const kda_desc *desc);
KDA_API int kda_prefill_backward(const kda_desc *desc,
                                 const void *q, const void *k, const void *v,
                                 const void *log_alpha, const void *beta,
                                 const int32_t *cu_seqlens, const float *initial_state,
                                 const void *d_out, const float *d_final_state,
                                 float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta,
                                 float *d_initial_state, kda_stream_t stream);

/*
 * One recurrent decode step for N independent sequences (deep dive section
 * 06, "fused recurrent KDA": decay, correct and write the state in place,
 * reading a fixed amount of memory per head).  Inputs are [N, H, *] (one
 * token per sequence, desc->total_tokens == N); state_inout fp32
 * [N, H, d_k, d_v] is read and overwritten in place; out [N, H, d_v].
 * No workspace is used (desc->workspace may be NULL).
 */
KDA_API int kda_decode_step(const kda_desc *desc,
                    const void *q, const void *k, const void *v,
                    const void *log_alpha, const void *beta,
                    float *state_inout, void *out, kda_stream_t stream);

/*
 * Synchronises `stream`, then returns the device status word that the last
 * kda_prefill on this workspace recorded: KDA_OK, KDA_ERR_BAD_SEQLENS,
 * KDA_ERR_BAD_SNAPSHOT or KDA_ERR_TIMEOUT (KDA_ERR_CUDA if the
 * synchronisation itself failed).
 */
KDA_API int kda_get_device_status(const kda_desc *desc, kda_stream_t stream);

/*
 * Size of the fixed scratch area kda_prefill_noalloc uses: 64 MiB.
 */
#define KDA_PREFILL_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * kda_prefill without a workspace, for callers that cannot allocate device
 * memory: code that gets all its buffers from someone else's pool, plugins
 * given only their inputs and outputs, or code where a cudaMalloc would
 * synchronise the device at the wrong moment.  The pages have no counterpart
 * to this call; it is a convenience of this library.
 *
 * Same arguments, layouts and results as kda_prefill; desc->workspace and
 * desc->workspace_bytes are ignored.  Instead the library's own static
 * device array of KDA_PREFILL_NOALLOC_SCRATCH_BYTES is used.  The runtime
 * reserves it on each device where this call is first used and holds it until
 * the process exits; no call allocates or frees anything.
 *  - Problems needing more scratch than that (kda_prefill_workspace_bytes
 *    larger than KDA_PREFILL_NOALLOC_SCRATCH_BYTES, for example more than about
 *    800 chunk-heads of 64 tokens on the bf16 head-size-128 path) are rejected
 *    with KDA_ERR_WORKSPACE before any GPU work.
 *  - Every call looks up the array's device address (cudaGetSymbolAddress,
 *    host-side, no stream work) with the caller's device current, so a
 *    context that was reset and re-created gets the new address.  The first
 *    call in a context may make the runtime load the library's kernels
 *    there: make it before any stream capture.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents (nothing in it needs to start at zero).  Calls whose GPU work
 *    may overlap -- different streams, or host threads without ordering --
 *    race on it and must be serialised by the caller.
 *  - The device status word lives in that array too; kda_get_device_status
 *    cannot read it.
 */
KDA_API int kda_prefill_noalloc(const kda_desc *desc,
                                const void *q, const void *k, const void *v,
                                const void *log_alpha, const void *beta,
                                const int32_t *cu_seqlens, const float *initial_state,
                                void *out, float *final_state, kda_stream_t stream);

/*
 * Diagnostic for the failure path: launches one CTA that waits on an mbarrier
 * no one ever arrives on, with the same bounded wait the prefill kernels use,
 * limited to timeout_ns (0 .. 1e9).  When the limit runs out the kernel stores
 * KDA_ERR_TIMEOUT in the device status word of desc->workspace and returns, so
 * kda_get_device_status then reports it.  Needs only desc->workspace (at least
 * 256 bytes); returns KDA_ERR_INVALID_ARGUMENT for a limit outside the range.
 */
KDA_API int kda_selftest_wait_timeout(const kda_desc *desc, int64_t timeout_ns, kda_stream_t stream);

/* Static, human-readable name of a status code. */
KDA_API const char *kda_status_string(int status);

/* The cudaError_t of the last failing CUDA call made by this thread (0 if none). */
KDA_API int kda_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */

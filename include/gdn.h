/*
 * gdn.h -- C ABI of libgdn: the gated delta-rule recurrence (Gated DeltaNet)
 * on one NVIDIA GB300 (sm_103a).
 *
 * Per (batch row b, value head h) the library runs, for every token t,
 *     S <- alpha_t * S                  decay                (S: fp32 [dv, dk])
 *     delta_t = beta_t * (v_t - S k_t)  with the decayed S
 *     S <- S + delta_t k_t^T            rank-1 update, S[i][j] += delta_t[i] k_t[j]
 *     o_t = S (scale * q_t)             readout with the updated S
 * Key/query heads are shared by groups of value heads (inverse GQA): value
 * head h reads key/query head h / (Hv / Hk).
 *
 * Conventions shared by every entry point
 *  - All data pointers are DEVICE pointers, owned by the caller.  The library
 *    allocates nothing, frees nothing and never synchronises: work is enqueued
 *    on `stream` (a cudaStream_t; NULL = the legacy default stream) and the
 *    call returns.  Buffers must stay alive until that work completes.
 *  - Layouts are dense, row-major, innermost dimension last:
 *      q, k        [total_T, Hk, dk]     (Hq must equal Hk)
 *      v, out      [total_T, Hv, dv]
 *      alpha, beta [total_T, Hv]         alpha is the decay itself, in (0, 1]
 *                                        (or its log, with GDN_ALPHA_LOG below)
 *      state       [N, Hv, dv, dk] fp32  (dk fastest)
 *    Rows are either uniform (cu_seqlens == NULL: row b owns tokens
 *    b*T .. b*T+T-1, total_T = B*T) or packed (cu_seqlens: int32 [B+1] on the
 *    device, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = total_T; the
 *    `T` argument is then total_T).  Token bounds read from cu_seqlens are
 *    clamped to [0, total_T] on the device.
 *  - q and k are used as given (already normalised) unless GDN_QK_L2NORM asks
 *    the kernel to normalise them (see "Input conventions"); `scale` then
 *    multiplies q.
 *  - Float pointers (q, k, v, out, alpha, beta, states, state_update,
 *    workspace) must be 16-byte aligned; int32 pointers 4-byte aligned.
 *  - Argument errors are reported synchronously, before anything is launched.
 *    Output buffers may not overlap inputs or each other (GDN_ERR_ALIAS),
 *    except where an entry point allows an exact in-place state.
 *  - A failed launch returns GDN_ERR_CUDA; the CUDA error is left for the
 *    caller's next cudaGetLastError.
 *  - Calls can be captured into CUDA graphs (tested for the decode,
 *    speculative-step and prefill calls; no such claim is made for
 *    gdn_prefill_chunked_noalloc).  The first call on a device
 *    that runs a given kernel sets that kernel's attributes (and the first
 *    call of all resolves the device error word): CUDA runtime calls, so make
 *    one call of each kind before stream capture starts.  Later calls only
 *    launch kernels.  The tensor-core prefill launches its second kernel as a
 *    programmatic dependent of its first (captured as a programmatic edge).
 *
 * Sources (page title, section):
 *  [P2] "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's
 *       AOTI CUDA backend" (executorch issue 23097), work list: chunked GDN
 *       prefill with explicit initial / final state, FP32 recurrence with
 *       BF16 weights, layout and gate/scaling conventions.
 *  [P3] "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
 *       (onnxruntime PR 32767), "Changes" and "Test Coverage":
 *       state_update_capacity, the [batch] capture_count input, the packed
 *       float32 state_update output, the clamped per-row prefix of decay /
 *       shared-key / delta factors that replay S = decay*S + outer(key, delta),
 *       inverse-GQA key sharing, state_update_active = 0 clearing the output.
 *  [P3-DF] same page, "DFlash2 Prerequisite": replay of compact state
 *       updates after partial draft acceptance.
 *  [P1] "Enable the native Kev example on the WebGPU backend" (executorch
 *       issue 23099): an immutable prefix snapshot reused across batches;
 *       repeated evaluations leave the prefix unchanged.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* negative size, Hq != Hk, Hv % Hk != 0, missing pointer */
    GDN_ERR_UNSUPPORTED = 2, /* valid, but no kernel for this dk / dv / chunk / dtype */
    GDN_ERR_ALIAS = 3,       /* an output overlaps an input or another output */
    GDN_ERR_ALIGN = 4,       /* a pointer breaks the alignment rule above */
    GDN_ERR_CUDA = 5,        /* a CUDA launch failed */
    GDN_ERR_TIMEOUT = 6,     /* a kernel gave up a bounded wait (see gdn_device_errors) */
    GDN_ERR_WORKSPACE = 7    /* workspace missing or smaller than required */
};

/* Storage types of q / k / v / out (dtype_qkv) and alpha / beta (dtype_gate). */
enum { GDN_F32 = 0, GDN_F16 = 1, GDN_BF16 = 2 };

/*
 * Input conventions ("gate/scaling conventions" of the layer feeding the
 * recurrence [P2]), OR'd into the dtype arguments of every entry point that
 * reads q / k / alpha / beta.  Without them, q and k arrive normalised, alpha
 * is the decay itself and beta the write strength.
 *  GDN_QK_L2NORM   in dtype_qkv:  q and k are L2-normalised per head inside
 *                  the kernel, x / sqrt(sum_j x_j^2 + 1e-6), before q is
 *                  multiplied by scale.
 *  GDN_ALPHA_LOG   in dtype_gate: alpha holds g = log(decay) (<= 0 expected);
 *                  the decay is e^g (the chunked form uses g directly).
 *  GDN_BETA_LOGIT  in dtype_gate: beta holds logits; beta = 1 / (1 + e^-x).
 * A capture stores the factors the recurrence actually used: the decay e^g
 * and the normalised key, so that a replay rebuilds the same state.
 */
#define GDN_QK_L2NORM 0x100
#define GDN_ALPHA_LOG 0x200
#define GDN_BETA_LOGIT 0x400

/* Slot width, in floats, of one captured token in `state_update`:
 * Hv decays, then Hk*dk keys, then Hv*dv deltas. */
#define GDN_STATE_UPDATE_SLOT(Hk, Hv, dk, dv) \
    ((size_t)(Hv) + (size_t)(Hk) * (dk) + (size_t)(Hv) * (dv))

/*
 * gdn_prefill_workspace_size -- bytes of device workspace that
 * gdn_prefill_chunked needs for these sizes (0 if none).  T as in
 * gdn_prefill_chunked; varlen != 0 when cu_seqlens will be passed.  The
 * tensor-core path (dk, dv in {32, 64, 128}, chunk 64, 16-bit q/k/v) stores
 * about 41 KB per (chunk, value head), plus, with packed rows, a table of
 * every row's first chunk and the order in which the carry takes the rows
 * (4 (2 B + 1) bytes rounded up to 1 KB).  dtype_qkv may carry the
 * GDN_QK_L2NORM bit (the same code as passed to the prefill; it does not
 * change the size).  Returns (size_t)-1 for invalid sizes or other flag bits.
 */
GDN_API size_t gdn_prefill_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv,
                                          int chunk, int dtype_qkv, int varlen);

/*
 * gdn_prefill_chunked -- chunked parallel prefill with explicit initial and
 * final state [P2].  Tokens are processed `chunk` at a time in the UT/WY
 * form of the recurrence; the last chunk of each row may be shorter (ragged
 * tail).  No capture: capture needs per-token transitions, which only
 * gdn_recurrent_capture emits [P3].
 *
 *  q, k, v, alpha, beta   inputs, layouts above (dtype_qkv / dtype_gate);
 *                         precondition: every alpha in (0, 1].
 *  cu_seqlens             NULL (uniform rows) or int32 [B+1], device.
 *  initial_state          NULL (start from zeros) or fp32 [num_initial_states, Hv, dv, dk].
 *  initial_state_indices  NULL (row b starts from state b; then
 *                         num_initial_states >= B) or int32 [B], device:
 *                         row b starts from state indices[b] (several rows may
 *                         share one read-only snapshot [P1]).  An index
 *                         outside [0, num_initial_states) starts that row from
 *                         zeros and sets GDN_DEVERR_BAD_INDEX.
 *  final_state            NULL (not written) or fp32 [B, Hv, dv, dk].  May be
 *                         exactly initial_state (in place) only when
 *                         initial_state_indices is NULL.  The initial state is
 *                         otherwise never written.
 *  out                    [total_T, Hv, dv], dtype_qkv, rounded to nearest even.
 *  chunk                  16, 32 or 64.
 *  workspace              device buffer of gdn_prefill_workspace_size() bytes
 *                         (may be NULL when that is 0); contents are scratch.
 */
GDN_API int gdn_prefill_chunked(const void *q, const void *k, const void *v,
                        const void *alpha, const void *beta,
                        const int32_t *cu_seqlens, const float *initial_state,
                        const int32_t *initial_state_indices,
                        int num_initial_states, float *final_state, void *out,
                        int B, int T, int Hq, int Hk, int Hv, int dk, int dv,
                        int chunk, float scale, int dtype_qkv, int dtype_gate,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_chunked_checkpoints -- gdn_prefill_chunked that also writes the
 * state at chunk boundaries, so that a prefix can later be resumed from any
 * of them (prefix-snapshot reuse at an offset [P1]: a snapshot is a state
 * after a prefix; here one is kept every L tokens).  Arguments shared with
 * gdn_prefill_chunked mean the same; gdn_prefill_chunked is this call with no
 * checkpoints.
 *
 *  checkpoint_interval    >= 1 chunks: boundaries every L = interval * chunk
 *                         tokens of each row.
 *  checkpoint_capacity    >= 0 slots per row (0: none, checkpoints may be NULL).
 *  checkpoints            fp32 [B, checkpoint_capacity, Hv, dv, dk] (output).
 *                         Slot j of row b holds the state after (j + 1) * L
 *                         tokens of the row, for
 *                         j < min(capacity, floor(T_b / L)); later slots are
 *                         not written (their contents are unspecified).  The
 *                         state past the last full boundary is final_state.
 */
GDN_API int gdn_prefill_chunked_checkpoints(const void *q, const void *k, const void *v,
                                            const void *alpha, const void *beta,
                                            const int32_t *cu_seqlens,
                                            const float *initial_state,
                                            const int32_t *initial_state_indices,
                                            int num_initial_states, float *final_state,
                                            void *out, int B, int T, int Hq, int Hk, int Hv,
                                            int dk, int dv, int chunk, float scale,
                                            int dtype_qkv, int dtype_gate, float *checkpoints,
                                            int checkpoint_capacity, int checkpoint_interval,
                                            void *workspace, size_t workspace_bytes,
                                            void *stream);

/*
 * gdn_prefill_chunked_capture -- gdn_prefill_chunked that also emits the
 * compact state-update capture of gdn_recurrent_capture (same arguments, same
 * slot layout, same clamp, same inactive behaviour).  The chunked form's
 * Delta rows are the tokens' deltas (the delta rule's delta, formed with the
 * decayed state), so the chunked path can emit them too; on the page the
 * chunked path emits none and capture forces the recurrent path [P3
 * "Changes"].  Accuracy of the captured deltas is that of the path: fp32
 * arithmetic on the CUDA-core path; on the tensor-core path (16-bit
 * operands) they carry the same relative error as its outputs.
 */
GDN_API int gdn_prefill_chunked_capture(const void *q, const void *k, const void *v,
                                        const void *alpha, const void *beta,
                                        const int32_t *cu_seqlens, const float *initial_state,
                                        const int32_t *initial_state_indices,
                                        int num_initial_states, float *final_state, void *out,
                                        int B, int T, int Hq, int Hk, int Hv, int dk, int dv,
                                        int chunk, float scale, int dtype_qkv, int dtype_gate,
                                        int state_update_capacity, const int32_t *capture_count,
                                        const int32_t *state_update_active,
                                        float *state_update, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * gdn_recurrent_capture -- per-token recurrent (decode / verify) path with
 * compact state-update capture [P3].  Arguments shared with
 * gdn_prefill_chunked mean the same (alpha = 0 is allowed here).
 *
 *  state_update_capacity  >= 0 slots per row; 0 disables capture.
 *  capture_count          int32 [B], device; required when capacity > 0.
 *                         Row b captures its first n_b tokens,
 *                         n_b = clamp(capture_count[b], 0, min(capacity, T_b)).
 *  state_update_active    NULL (active) or a device int32 scalar, read by the
 *                         kernel (so a captured CUDA graph can flip it).
 *  state_update           fp32 [B, capacity, GDN_STATE_UPDATE_SLOT(Hk,Hv,dk,dv)].
 *                         Slot t of row b holds token t's decay alpha of every
 *                         value head, key k of every key head (as fp32), and
 *                         delta of every value head.  While active, slots
 *                         t >= n_b are not written (their contents are
 *                         unspecified); while inactive (*active == 0) the whole
 *                         buffer is set to 0.0f and the recurrence still runs.
 */
GDN_API int gdn_recurrent_capture(const void *q, const void *k, const void *v,
                          const void *alpha, const void *beta,
                          const int32_t *cu_seqlens, const float *initial_state,
                          const int32_t *initial_state_indices,
                          int num_initial_states, float *final_state, void *out,
                          int B, int T, int Hq, int Hk, int Hv, int dk, int dv,
                          float scale, int dtype_qkv, int dtype_gate,
                          int state_update_capacity, const int32_t *capture_count,
                          const int32_t *state_update_active,
                          float *state_update, void *stream);

/*
 * gdn_replay_state_updates -- rebuild the state reached after an accepted
 * prefix [P3-DF]: for t < m_b, S <- decay_t * S + outer(delta_t, key_t)
 * (S[i][j] = decay * S[i][j] + delta[i] * key[j]), where
 * m_b = clamp(accepted_count[b], 0, capacity) and the factors are slot t of
 * row b of a state_update buffer written by gdn_recurrent_capture.
 * Precondition: m_b <= the n_b that capture used (later slots are unspecified).
 *
 *  state_in, state_out    fp32 [B, Hv, dv, dk]; state_out may equal state_in
 *                         exactly (in place); any other overlap is an error.
 *  state_update           fp32 [B, capacity, slot] (input).
 *  accepted_count         int32 [B], device.
 */
GDN_API int gdn_replay_state_updates(const float *state_in, float *state_out,
                             const float *state_update, int state_update_capacity,
                             const int32_t *accepted_count, int B, int Hk,
                             int Hv, int dk, int dv, void *stream);

/*
 * gdn_replay_verify -- one speculative-decoding step in one launch: replay
 * the accepted prefix of the previous verify pass, then verify the next
 * draft tokens [P3-DF: the DFlash2 loop is capture during verification,
 * replay of the accepted prefix, and a state that must match the
 * non-speculative run].  It equals gdn_replay_state_updates followed by
 * gdn_recurrent_capture, but reads each state once and writes it once instead
 * of reading it twice and writing it once.  Per (row b, value head h):
 *     S  = state_in[b]                        (zeros when state_in is NULL)
 *     for t < m_b: S <- decay_t * S + outer(delta_t, key_t)
 *                  factors from slot t of prev_state_update, row b;
 *                  m_b = clamp(accepted_count[b], 0, prev_capacity)
 *     state_out[b] = S                        (the committed state)
 *     then the row's T_b draft tokens run from S exactly as in
 *     gdn_recurrent_capture: out, capture into state_update, and the state
 *     after the last draft token in draft_final_state (if not NULL).
 *
 *  q ... beta, cu_seqlens   the draft tokens, as in gdn_recurrent_capture;
 *                         rows with T_b = 0 only replay.
 *  state_in               NULL or fp32 [B, Hv, dv, dk] (no index gather).
 *  state_out              fp32 [B, Hv, dv, dk], required; may be exactly
 *                         state_in (in place: rows with m_b = 0 are then not
 *                         rewritten).
 *  prev_state_update      fp32 [B, prev_capacity, slot], the previous call's
 *                         capture (input); NULL allowed when prev_capacity == 0
 *                         (nothing is replayed).  It must not overlap
 *                         state_update: alternate two capture buffers.
 *  accepted_count         int32 [B], device; required when prev_capacity > 0.
 *                         Precondition: m_b <= the n_b the capture used.
 *  draft_final_state      NULL or fp32 [B, Hv, dv, dk] (output).
 *  state_update_capacity, capture_count, state_update_active, state_update
 *                         the new capture, as in gdn_recurrent_capture.
 */
GDN_API int gdn_replay_verify(const void *q, const void *k, const void *v,
                              const void *alpha, const void *beta,
                              const int32_t *cu_seqlens, const float *state_in,
                              float *state_out, const float *prev_state_update,
                              int prev_capacity, const int32_t *accepted_count,
                              float *draft_final_state, void *out, int B, int T, int Hq,
                              int Hk, int Hv, int dk, int dv, float scale, int dtype_qkv,
                              int dtype_gate, int state_update_capacity,
                              const int32_t *capture_count,
                              const int32_t *state_update_active, float *state_update,
                              void *stream);

/*
 * gdn_prefill_chunked_noalloc -- gdn_prefill_chunked for callers that cannot
 * allocate device memory: runtimes with their own memory planner that forbid
 * hidden allocations, or latency-critical paths that must never enter the
 * allocator.  Same arguments and results as
 * gdn_prefill_chunked, without the workspace: the library uses a fixed device
 * buffer of GDN_NOALLOC_SCRATCH_BYTES compiled into it (every device that
 * loads the library keeps it until the process exits).  The pages describe
 * no such entry point; it exists only for these callers.
 *
 *  - Sizes: the call is accepted when gdn_prefill_workspace_size(...) for the
 *    same arguments is <= GDN_NOALLOC_SCRATCH_BYTES (32 MiB: e.g. up to 799
 *    (chunk, value head) records on the tensor-core path, 1536 tokens at
 *    Hv = 32 in one row); larger problems return GDN_ERR_WORKSPACE before
 *    anything is launched.  Shapes that need no workspace always fit.
 *  - The first call on a device looks up the buffer's device address (a CUDA
 *    runtime query, cached per device); make that first call before any
 *    stream capture starts.
 *  - All calls share the buffer and it keeps the last call's contents (the
 *    prefill writes every scratch byte it reads, so nothing is cleared).
 *    Calls whose GPU work overlaps (e.g. on unordered streams) race on it:
 *    serialise them.
 *  - No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
GDN_API int gdn_prefill_chunked_noalloc(const void *q, const void *k, const void *v,
                                        const void *alpha, const void *beta,
                                        const int32_t *cu_seqlens, const float *initial_state,
                                        const int32_t *initial_state_indices,
                                        int num_initial_states, float *final_state, void *out,
                                        int B, int T, int Hq, int Hk, int Hv, int dk, int dv,
                                        int chunk, float scale, int dtype_qkv, int dtype_gate,
                                        void *stream);

/* Device-side error bits (gdn_device_errors). */
enum {
    GDN_DEVERR_BAD_INDEX = 1, /* an initial_state_indices entry was out of range */
    GDN_DEVERR_TIMEOUT = 2    /* a kernel abandoned a bounded wait */
};

/*
 * gdn_device_errors -- synchronises `stream`, then returns in *flags the
 * GDN_DEVERR_* bits that kernels on the current device raised since the
 * last call, and clears them.  Returns GDN_ERR_TIMEOUT if the timeout bit was
 * set, GDN_ERR_CUDA on a CUDA failure, else GDN_OK.
 */
GDN_API int gdn_device_errors(void *stream, uint32_t *flags);

/*
 * gdn_set_wait_limit_ns -- testing hook for the failure path.  Every kernel
 * bounds its waits on another warp's work (pipeline hand-offs inside a CTA);
 * a wait that runs out sets GDN_DEVERR_TIMEOUT, the CTA waits (with the full
 * limit) for its own copies in flight, releases its tensor memory and exits,
 * and gdn_device_errors then returns GDN_ERR_TIMEOUT.  The limit is 1 s by
 * default; this sets it, for calls made afterwards from any thread, to `ns`
 * nanoseconds (0 restores the default).  A limit below 1000 ns gives up at
 * the first check that finds a hand-off incomplete, which lets a test drive
 * the timeout path on a small case.  Results of a call whose wait ran out
 * are unspecified.  Not meant for production use.
 */
GDN_API void gdn_set_wait_limit_ns(uint64_t ns);

/* Human-readable text for a status code (static storage). */
GDN_API const char *gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */

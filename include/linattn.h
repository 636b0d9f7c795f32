/*
 * linattn.h -- C ABI of the GB300 (sm_103a) causal linear-attention library.
 *
 * The operations follow the web page "From GPT-2 to Kimi K3, explained"
 * (sections Linear attention; DeltaNet (Fast Weight Programmers);
 * DeltaNet (Parallelizing Linear Transformers with Delta Rule); Gated
 * DeltaNet; KDA / Kimi Linear).  Each head keeps a fixed dk x dv fp32 state
 * S instead of a growing KV cache.
 *
 * Conventions shared by every call
 * --------------------------------
 * - State layout: row convention of the page's listings, S in R^{dk x dv},
 *   read o = S^T q, write S += k u^T.  States are fp32, row-major,
 *   [N][H][dk][dv] (the column form S_t q_t of the chunkwise section is its
 *   transpose; outputs are identical).
 * - Token tensors are packed, all sequences back to back:
 *   q, k [ntok][H][dk]; v, o [ntok][H][dv]; beta_logits [ntok][H];
 *   gate_logits [ntok][H][dk].  All are dense and contiguous, in the I/O
 *   dtype `io` (LA_F32 or LA_BF16); states are always fp32.
 * - cu_seqlens: int32 DEVICE array of N+1 non-decreasing offsets into the
 *   token dimension; sequence n owns tokens [cu_seqlens[n], cu_seqlens[n+1]).
 *   An equal-length batch of B sequences of T tokens is {0, T, 2T, ..., BT}.
 *   ntok is the number of packed tokens the token tensors hold (their first
 *   dimension); every cu_seqlens entry must lie in [0, ntok].
 *   cu_seqlens_host (nullable) is a HOST copy of the same array; when given,
 *   it is validated before any launch.  Without it, a device-side range
 *   check skips offending sequences and la_check_device reports
 *   LA_ERR_INVALID_ARG.
 * - Supported head sizes: dk, dv in {64, 128}.  N >= 1, H >= 1.
 * - Every pointer is a device pointer unless stated otherwise.  The caller
 *   owns every buffer; the library allocates, frees and synchronises nothing
 *   (except la_check_device, which synchronises the given stream, and the
 *   static buffer of la_prefill_delta_static described there).  Outputs
 *   must not alias inputs; final states may alias the matching initial state
 *   only where stated.
 * - stream: a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  All work is enqueued on it; calls return once enqueued.
 * - Errors: every call returns an la_status.  Argument checks run on the
 *   host before any launch, and a rejected call launches nothing.  A launch
 *   failure returns LA_ERR_CUDA.  No C++ exception crosses this boundary.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1, /* null pointer, bad size, non-monotone cu_seqlens_host, bad flag */
    LA_ERR_UNSUPPORTED = 2, /* valid request this build has no kernel for (e.g. dk = 96)     */
    LA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed                            */
    LA_ERR_TIMEOUT = 4,     /* a bounded in-kernel wait expired (reported by la_check_device)  */
    LA_ERR_TOO_LARGE = 5    /* la_prefill_delta_static: scratch need above its static buffer   */
} la_status;

typedef enum la_dtype { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* Prologue options (`flags`) for the delta-rule calls.
 * LA_L2NORM_K: k <- k / max(||k||_2, 1e-12) per token and head.
 * LA_L2NORM_Q: the same for q.
 * LA_SILU_QK : q, k <- silu(q), silu(k), applied before the normalisation
 *              (the page's DeltaNet layer applies silu, then the L2
 *              normalisation). */
#define LA_L2NORM_K 1u
#define LA_L2NORM_Q 2u
#define LA_SILU_QK 4u
/* LA_GATE_SCALAR: gate_logits holds one value per token and head
 * ([ntok][H] in prefill, [N][H] in decode) and alpha applies to every key
 * channel alike -- the scalar decay of section Gated DeltaNet (Mamba-2's
 * S_t = alpha_t S_{t-1} + k_t v_t^T) instead of the per-key-channel decay of
 * section KDA / Kimi Linear.  Requires gate_logits. */
#define LA_GATE_SCALAR 8u
/* LA_ADDITIVE: the decayed additive state of section Gated DeltaNet
 * (Mamba-2: S_t = alpha_t S_{t-1} + k_t v_t^T, the new association added at
 * full strength): u_t = v_t, no read of the old value and no beta, so
 * S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T.  Any gate form (none, per key
 * channel, LA_GATE_SCALAR) applies; beta_logits is ignored and may be NULL.
 * Accepted by la_prefill_delta(_static), la_decode_step(_slots) and
 * la_backward_delta (which then writes d_beta_logits = 0). */
#define LA_ADDITIVE 16u

/* Causal ELU+1 linear attention, chunkwise-parallel prefill.
 * Defined in section Linear attention (the forward() that replaces the KV
 * cache) and its chunked form in section DeltaNet (Parallelizing Linear
 * Transformers with Delta Rule):
 *   phi(x) = elu(x) + 1 on q and k separately;
 *   S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *   o_t = S_t^T phi(q_t) / (z_t^T phi(q_t)).
 * init_S [N][H][dk][dv], init_z [N][H][dk]: nullable (NULL = zero state).
 * final_S, final_z: nullable outputs, same shapes; final_S may equal init_S
 * and final_z may equal init_z (in-place continuation). */
la_status la_prefill_linear(const void *q, const void *k, const void *v, void *o, la_dtype io,
                            const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                            int ntok, int H, int dk, int dv, const float *init_S,
                            const float *init_z, float *final_S, float *final_z, void *stream);

/* (Gated) delta rule, chunkwise-parallel prefill.
 * Defined in sections DeltaNet (Fast Weight Programmers) (the step), DeltaNet
 * (Parallelizing Linear Transformers with Delta Rule) (the Householder
 * reparametrisation and the chunkwise WY/UT algorithm, eq. 8-10), Gated
 * DeltaNet (decay alpha, cumulative decay) and KDA / Kimi Linear (one decay
 * per key channel).  Per sequence and head, with S' = Diag(alpha_t) S_{t-1}:
 *   u_t = beta_t (v_t - S'^T k_t),  S_t = S' + k_t u_t^T,  o_t = scale S_t^T q_t
 * where beta_t = sigmoid(beta_logits[t][h]) and
 * alpha_t[c] = exp(-softplus(gate_logits[t][h][c])).
 * gate_logits: nullable; NULL means alpha = 1 (plain DeltaNet).  With
 * LA_GATE_SCALAR it is [ntok][H] and alpha_t applies to all channels.
 * flags: LA_L2NORM_K | LA_L2NORM_Q | LA_SILU_QK | LA_GATE_SCALAR | LA_ADDITIVE
 * (above).
 * chunk: tokens per chunk of the state recurrence, 64 or 128 (the page
 * names both as the usual sizes).  128 needs io = LA_BF16 and dk = dv = 64
 * (else LA_ERR_UNSUPPORTED): the chunk-parallel pass still forms the UT/WY
 * operands per 64 tokens, and the recurrence joins each pair of them into
 * the 128-token chunk's operands (the off-diagonal block of a two-level
 * blocked solve) before its step, so the sequential chain runs once per 128
 * tokens.  The results agree with chunk 64 up to rounding.
 * scale: output scale (the page's delta-rule listings use 1.0).
 * init_S: nullable [N][H][dk][dv]; final_S: nullable, may equal init_S.
 * workspace / workspace_bytes: device scratch of at least
 * la_prefill_delta_workspace_size(...) bytes, 256-byte aligned; may be NULL
 * only when that size is 0 (else LA_ERR_INVALID_ARG, nothing launched).  It
 * needs no initialisation and holds nothing useful afterwards; calls that
 * may run at the same time (other streams) need separate workspaces. */
la_status la_prefill_delta(const void *q, const void *k, const void *v, const void *beta_logits,
                           const void *gate_logits, void *o, la_dtype io,
                           const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                           int ntok, int H, int dk, int dv, int chunk, float scale,
                           unsigned flags, const float *init_S, float *final_S, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Scratch bytes la_prefill_delta needs for these sizes; ntok = total packed
 * tokens.  Nonzero exactly for the tensor-core configurations (io = LA_BF16,
 * dk = dv in {64, 128}, chunk = 64; or dk = dv = 64, chunk = 128, which
 * needs the same bytes), whose first pass computes everything
 * that depends on one chunk alone (the WY/UT operands of eq. 10 and the
 * decayed q, k of the chunk) for all chunks in parallel and hands it to the
 * sequential state pass through this buffer: 8 bytes per chunk slot (a
 * chunk table, filled only by la_backward_delta's forward pass), then one
 * record per (chunk slot, head) of 41 KB (d = 64) or 73 KB (d = 128), with
 * at most ntok/64 + N + 1 slots, then a 4-byte flag per record and 256
 * bytes of task counters (used when both passes run in one launch, d = 64).
 * 0 otherwise. */
size_t la_prefill_delta_workspace_size(int N, int ntok, int H, int dk, int dv, int chunk,
                                       la_dtype io);

/* Number of kernels one la_prefill_delta call with these sizes and options
 * launches on the current device, given 16-byte-aligned tensors and a
 * workspace of la_prefill_delta_workspace_size bytes (has_gate: whether
 * gate_logits is given): 2 on the tensor-core configurations
 * (chunk-parallel kernel, then the recurrence kernel), 1 on the CUDA-core
 * path; 0 if la_prefill_delta would reject the arguments.  (A one-launch
 * form for d = 64 -- one cooperative kernel running both passes, after a
 * memset of the workspace's flags -- is built but not dispatched; this
 * query would report 1 for the calls it would take.)  For planning (graph capture, launch accounting);
 * the page has no counterpart. */
int la_prefill_delta_launches(int N, int ntok, int H, int dk, int dv, int chunk, la_dtype io,
                              unsigned flags, int has_gate);

/* la_prefill_delta without a caller workspace, allocating nothing: the
 * per-chunk scratch comes from one library-owned static device buffer of
 * LA_STATIC_SCRATCH_BYTES (256 MiB) per device.  The page has no counterpart:
 * it is a deployment convenience (CUDA-graph capture, or callers without an
 * allocator), not part of the method.
 * Arguments, results and errors are those of la_prefill_delta, plus
 * LA_ERR_TOO_LARGE (nothing launched) when la_prefill_delta_workspace_size
 * for these sizes exceeds LA_STATIC_SCRATCH_BYTES (e.g. the d = 64 layout
 * fits about 6000 chunk-heads: ntok/64 + N + 1 slots times H).
 * The buffer's address is looked up (cudaGetSymbolAddress) on the first call
 * on each device; make that first call outside CUDA stream capture.  The
 * buffer needs no initialisation (every call rewrites what it reads).  All
 * calls on a device share it, so calls whose executions may overlap in time
 * (different streams, or host threads without ordering) race on it and give
 * undefined results: serialise them.
 * Footprint: the buffer sits in a CUDA module of its own.  Under lazy module
 * loading (the CUDA runtime's default) it is reserved on a device at the
 * first la_prefill_delta_static call there and held until the process
 * exits; processes that never call this entry point never reserve it.
 * Under eager loading (CUDA_MODULE_LOADING=EAGER) every device the process
 * initialises reserves it at context creation. */
#define LA_STATIC_SCRATCH_BYTES (256u << 20)
la_status la_prefill_delta_static(const void *q, const void *k, const void *v,
                                  const void *beta_logits, const void *gate_logits, void *o,
                                  la_dtype io, const int32_t *cu_seqlens,
                                  const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                                  int dv, int chunk, float scale, unsigned flags,
                                  const float *init_S, float *final_S, void *stream);

/* One recurrent decode step: one new token for each of N sequences, state
 * updated IN PLACE (sections DeltaNet (Fast Weight Programmers) and Gated
 * DeltaNet: forward(x, cache) with t = 1; KDA / Kimi Linear for the
 * per-channel decay).  Same arithmetic as la_prefill_delta with one token:
 *   S' = Diag(alpha) S;  u = beta (v - S'^T k);  S <- S' + k u^T;
 *   o = scale S^T q.
 * q, k [N][H][dk]; v, o [N][H][dv]; beta_logits [N][H];
 * gate_logits [N][H][dk] ([N][H] with LA_GATE_SCALAR) or NULL (alpha = 1);
 * state [N][H][dk][dv] fp32,
 * read and rewritten once per call.  state must not alias any other buffer. */
la_status la_decode_step(const void *q, const void *k, const void *v, const void *beta_logits,
                         const void *gate_logits, void *o, la_dtype io, int N, int H, int dk,
                         int dv, float scale, unsigned flags, float *state, void *stream);

/* la_decode_step over a pool of states addressed through a slot map, for
 * servers that keep the recurrent states of many requests in one
 * persistent buffer and step an arbitrary subset of them.  The page has no
 * counterpart (its forward(x, cache) takes each sequence's cache on its
 * own); the arithmetic per sequence is exactly that of la_decode_step.
 * state_pool [n_slots][H][dk][dv] fp32; state_indices: device int32 [N],
 * sequence n reads and rewrites state_pool[state_indices[n]] in place.
 * A negative index marks a padding sequence: its state and its output rows
 * are left untouched.  Non-negative indices must be distinct (two
 * sequences on one slot race; not checked).  An index >= n_slots touches
 * nothing for that sequence and makes the next la_check_device return
 * LA_ERR_INVALID_ARG.  Other arguments and errors as la_decode_step, plus
 * LA_ERR_INVALID_ARG for a NULL state_indices or n_slots < 1. */
la_status la_decode_step_slots(const void *q, const void *k, const void *v,
                               const void *beta_logits, const void *gate_logits, void *o,
                               la_dtype io, int N, int H, int dk, int dv, float scale,
                               unsigned flags, float *state_pool, int n_slots,
                               const int32_t *state_indices, void *stream);

/* Gradients of la_prefill_delta (the page gives the forward pass only; its
 * section DeltaNet (Parallelizing Linear Transformers with Delta Rule)
 * motivates the chunked form by training).  Given the gradient d_o of the
 * outputs o (and optionally d_final_S of the final states), returns the
 * gradients of the loss with respect to every input of the forward call
 * with the same q, k, v, beta_logits, gate_logits, cu_seqlens, scale, flags
 * and init_S: the chain rule through each step of the token recurrence in
 * reverse and through the prologue (sigmoid, -softplus, silu, L2 norm).
 * Inputs as la_prefill_delta; d_o [ntok][H][dv] in the I/O dtype;
 * d_final_S [N][H][dk][dv] fp32 or NULL (zero).  Outputs, all fp32, shaped
 * like their inputs: dq, dk [ntok][H][dk]; dv [ntok][H][dv];
 * d_beta_logits [ntok][H]; d_gate_logits like gate_logits (required iff
 * gate_logits is given); d_init_S [N][H][dk][dv] or NULL.  Rows of tokens
 * outside every sequence are not written.
 * Workspace: la_backward_delta_workspace_size bytes, 256-byte aligned
 * (the forward pass's per-chunk records, the state and its gradient at
 * every chunk start, du per chunk; or, token-serial, checkpoints and
 * per-token column sums); LA_ERR_INVALID_ARG if smaller or missing.
 * dk, dv in {64, 128}.  Two forms, chosen from the arguments: chunkwise
 * (io = LA_BF16, dk = dv, every tensor 16-byte aligned; any gate, either
 * update rule) -- the tensor-core forward pass, a reverse pass over the
 * chunks for the state gradient (tensor cores, the gradient held in tensor
 * memory), then every (chunk, head) in parallel; token-serial otherwise.
 * Sums over value columns inside a thread block use shared-memory atomics,
 * so the last bits of dq, dk, d_beta_logits and d_gate_logits may differ
 * between runs. */
size_t la_backward_delta_workspace_size(int N, int ntok, int H, int dk, int dv);
la_status la_backward_delta(const void *q, const void *k, const void *v, const void *beta_logits,
                            const void *gate_logits, const void *d_o, const float *d_final_S,
                            la_dtype io, const int32_t *cu_seqlens,
                            const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                            int dv, float scale, unsigned flags, const float *init_S, float *dq,
                            float *dk_out, float *dv_out, float *d_beta_logits,
                            float *d_gate_logits, float *d_init_S, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Training pair: the forward pass that keeps what the gradients need, and
 * the gradients without recomputing that forward.  (The page motivates the
 * chunked form by training, section DeltaNet (Parallelizing Linear
 * Transformers with Delta Rule); it has no such interface.  la_backward_delta
 * runs the forward again inside the call; a training step that has just run
 * it pays for it twice.)
 *
 * la_prefill_delta_train: the outputs of la_prefill_delta at chunk = 64 (o,
 * and final_S when given), from the same tensor-core kernels, plus the
 * per-chunk records, each chunk's T = (I + A)^{-1} and the fp32 state at
 * every chunk start, kept in `saved`: a buffer of
 * la_backward_delta_workspace_size(N, ntok, H, dk, dv) bytes, 256-byte
 * aligned, owned by the caller and left untouched by the library between the
 * two calls.  Arguments otherwise as la_prefill_delta.  Configurations: those
 * of the chunkwise backward (io = LA_BF16, dk = dv in {64, 128}, every tensor
 * 16-byte aligned); LA_ERR_UNSUPPORTED otherwise (use la_prefill_delta and
 * la_backward_delta there); LA_ERR_INVALID_ARG for a missing, small or
 * misaligned `saved`. */
la_status la_prefill_delta_train(const void *q, const void *k, const void *v,
                                 const void *beta_logits, const void *gate_logits, void *o,
                                 la_dtype io, const int32_t *cu_seqlens,
                                 const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                                 int dv, float scale, unsigned flags, const float *init_S,
                                 float *final_S, void *saved, size_t saved_bytes, void *stream);

/* la_backward_delta_saved: the gradients of la_backward_delta, with the same
 * arguments and outputs, taking the forward's tensors from `saved` as the
 * preceding la_prefill_delta_train left them (pass that call's q, k, v,
 * beta_logits, gate_logits, cu_seqlens, scale, flags and init_S; the results
 * are undefined otherwise, though every access stays inside the given
 * tensors).  The reverse chain and the per-chunk kernels read `saved` and
 * write only its scratch part (dS' and du of every chunk), so the call may be
 * repeated on the same saved tensors.  If the gradient tensors are not all
 * 16-byte aligned, it runs la_backward_delta's token-serial form instead,
 * which recomputes the forward in the same buffer. */
la_status la_backward_delta_saved(const void *q, const void *k, const void *v,
                                  const void *beta_logits, const void *gate_logits,
                                  const void *d_o, const float *d_final_S, la_dtype io,
                                  const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                  int N, int ntok, int H, int dk, int dv, float scale,
                                  unsigned flags, const float *init_S, float *dq, float *dk_out,
                                  float *dv_out, float *d_beta_logits, float *d_gate_logits,
                                  float *d_init_S, void *saved, size_t saved_bytes, void *stream);

/* Synchronises `stream`, then reports (and clears) any error raised on the
 * current device since the previous check: LA_ERR_TIMEOUT if a bounded
 * in-kernel wait gave up, LA_ERR_INVALID_ARG if a kernel found cu_seqlens
 * or a state slot out of range, LA_ERR_CUDA for a CUDA error, else LA_OK. */
la_status la_check_device(void *stream);

/* Self-test of the failure path (no computation): launches one kernel on
 * `stream` that waits on an mbarrier nothing ever completes.  The wait is
 * bounded like every in-kernel wait of the library; when it runs out (well
 * under a second) the kernel records a timeout in the device error word and
 * ends normally, so the next la_check_device returns LA_ERR_TIMEOUT and the
 * context stays usable.  Returns LA_ERR_CUDA if the launch fails, else
 * LA_OK (the timeout itself is reported by la_check_device). */
la_status la_selftest_wait_timeout(void *stream);

/* Static, human-readable name of a status code. */
const char *la_status_string(la_status s);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */

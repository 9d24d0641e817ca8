/*
 * gdn.h -- C ABI of the chunked Gated DeltaNet (gated delta rule) forward and
 * backward for NVIDIA GB300 (sm_103a).
 *
 * The operation.  Per batch row b and value head j (key head kh = j / (Hv/Hk)),
 * with the state written transposed, h = S^T of shape d_k x d_v:
 *     h_t = exp(g_t) (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T,
 *     o_t = h_t^T q_t,          h_{-1} = h0,  hT = h_{T-1}.
 * It is evaluated in chunks of `chunk` tokens through the WY/UT form: per chunk
 * the UT inverse T = (I + S)^-1 of S = tril(diag(beta) (K K^T * decay), -1)
 * (blockwise doubling ladder), w = T diag(beta exp(G)) K, u = T diag(beta) V,
 * the inter-chunk step h' = (exp(g_last) I - k_g^T w) h + k_g^T u = A h + B,
 * and the masked intra-chunk output.  Sources (pages' titles and sections):
 *   - the inter-chunk step as an affine map h' = A h + B and the composition
 *     law (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2): issue "GatedDeltaNet does
 *     not support ici_context_parallelism", section "The recurrence is affine,
 *     so it can be parallelized";
 *   - the two-pass scan (fold each stretch of chunks into one (A, B), exclusive
 *     prefix, replay from the incoming state): PR "Shard the GatedDeltaNet
 *     sequence under ici_context_parallelism", description;
 *   - the ladder inverse, its analytic backward dS = -(T^T dT T^T) (strictly
 *     lower), the reverse chunk walk of the backward and initial/final state
 *     as first-class inputs/outputs: PR "Fuse the Gated Delta Net inter-chunk
 *     scan into a Pallas TPU kernel", section "Changes".
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers (cudaMalloc'd, or any memory the device can
 *     address), contiguous, 16-byte aligned.  bf16 tensors are passed as
 *     void* to raw IEEE bfloat16 data.  The caller owns all memory; the
 *     library allocates nothing, keeps no state between calls and never
 *     synchronises the stream -- except gdn_chunk_fwd_noalloc, whose fixed
 *     scratch array (in the library's device image) and per-device address
 *     cache persist between calls (see its declaration), and the status
 *     readers, which synchronise.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *     is enqueued on it asynchronously; outputs are valid once it has run.
 *   - Layouts: q, k [B, T, Hk, d_k]; v, o, dO, dv [B, T, Hv, d_v];
 *     g, beta, dg, dbeta [B, T, Hv]; h0, hT, dhT, dh0 [B, Hv, d_k, d_v];
 *     dq, dk [B, T, Hk, d_k].
 *   - Return value: GDN_OK, or a negative gdn_status.  Argument errors are
 *     detected on the host before anything is enqueued, so a failed call has
 *     no effect.  GDN_ERR_CUDA reports a launch failure (cudaGetLastError).
 *   - Supported sizes in this version: d_k = d_v = 128, chunk = 128, any
 *     T >= 0 (a ragged last chunk is zero-padded with g = 0, beta = 0, which
 *     leaves the state unchanged), Hv a multiple of Hk.  The forward entry
 *     points (gdn_chunk_fwd, its _timed and _ex variants without a saved
 *     buffer, gdn_chunk_fwd_noalloc, gdn_segment_fold, gdn_layer_fwd,
 *     gdn_debug_ut and their workspace sizes) also take chunk = 64 (PR "Shard
 *     the GatedDeltaNet sequence under ici_context_parallelism", review
 *     thread: forming each device's A_loc with 64-token chunks): the state
 *     then steps every 64 tokens.  The backward entry points, and a forward
 *     that keeps tiles for them, take chunk = 128 only (GDN_ERR_SHAPE
 *     otherwise); their results do not depend on the chunk size beyond
 *     rounding, so a backward with chunk = 128 serves a forward run with 64.
 *   - Workspace: the caller passes `ws` of at least the size the matching
 *     *_workspace_bytes call returns for the same arguments (256-byte aligned).
 *     Its contents on entry do not matter.  Its first 4 bytes are a status
 *     word: the call clears it, and a kernel sets bit 0 if one of its bounded
 *     waits gives up (gdn_workspace_status reads it).
 *   - Bounded waits: the kernels wait only inside one block (for their TMA
 *     copies, their tensor-core products and hand-offs between their warps);
 *     every such wait gives up after 2e9 SM cycles (about one second), so
 *     a fault can leave wrong outputs and a set status bit but never a hung
 *     GPU.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_ARG = -1,        /* null required pointer, misalignment, Hv % Hk != 0, negative size */
  GDN_ERR_SHAPE = -2,      /* unsupported d_k, d_v or chunk */
  GDN_ERR_WORKSPACE = -3,  /* workspace missing or smaller than required */
  GDN_ERR_CUDA = -4,       /* a kernel launch failed */
  GDN_ERR_TIMEOUT = -5,    /* a bounded in-kernel wait gave up (see gdn_workspace_status) */
  GDN_ERR_UNSUPPORTED = -6 /* device is not sm_103 / sm_100 class */
} gdn_status;

/* Human-readable text of a status code (static storage, never NULL). */
const char* gdn_strerror(int status);

/* Number of chunk segments the forward/backward use when n_segments == 0: one
 * when the chunks are few or the batch rows and value heads already keep a
 * quarter of the SMs busy with the one-segment walk (4 CTAs each), else enough
 * segments to fill the SMs about twice with the segment fold (8 CTAs per
 * segment and head), at least 8 chunks each. */
int gdn_default_segments(int B, int T, int Hv, int chunk);

/*
 * Workspace bytes of gdn_chunk_fwd / gdn_chunk_bwd for these arguments
 * (n_segments as it will be passed, 0 = automatic).  Returns 0 for invalid
 * sizes.
 */
size_t gdn_fwd_workspace_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk,
                               int n_segments);
size_t gdn_bwd_workspace_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk,
                               int n_segments);

/*
 * Forward.  Reads q, k, v (bf16), g, beta (fp32, g is the per-token log-gate,
 * exp(g) the decay), h0 (fp32, NULL = zero state); writes o (bf16) and hT
 * (fp32, NULL = not written).
 * n_segments: 1 = one sequential walk over the chunks per (b, value head);
 * S > 1 = the two-pass segment scan with S segments of whole chunks (segment
 * s holds chunks [floor(sN/S), floor((s+1)N/S)) of the N chunks); 0 = the
 * library's choice (gdn_default_segments).  Results agree across segment
 * counts up to rounding.
 */
int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta, const float* h0, void* o, float* hT, int B, int T,
                  int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                  size_t ws_bytes, void* stream);

/*
 * Backward of gdn_chunk_fwd.  Takes the forward's inputs plus the output
 * cotangent dO (bf16, required) and the final-state cotangent dhT (fp32,
 * NULL = zero).  Writes dq, dk (bf16, summed over the value heads that share
 * each key head), dv (bf16), dg, dbeta (fp32) and dh0 (fp32, NULL = not
 * written).  The forward states are recomputed (nothing is saved from the
 * forward call).  n_segments as for the forward (it segments the reverse walk
 * of the state cotangent and the recomputation of the states).
 */
int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta, const float* h0, const void* dO, const float* dhT,
                  void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0, int B,
                  int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                  size_t ws_bytes, void* stream);

/*
 * Keeping the forward's per-chunk quantities for the backward.  The backward
 * needs, per chunk, the forward's w, u, P and the UT inverse T; gdn_chunk_bwd
 * recomputes them (one launch of the preparation).  A training step that runs
 * the backward of the same inputs right after the forward can instead let the
 * forward keep them in a caller buffer `saved` of gdn_saved_bytes bytes (w, u,
 * P, T, the state entering every chunk and Delta = u - w h, bf16,
 * [B, Hv, ceil(T/chunk), 128, 128] each, and with segments the state entering
 * every segment, fp32 [B, Hv, S, 128, 128]) and pass it to the backward, which
 * then skips the preparation and the recompute of the states (and, with
 * segments, the fold and prefix that recompute the segments' entering states):
 * it runs the reverse walk of the state cotangent and the gradients only.  The pages' own fused kernel
 * keeps the inverse for its backward in the same way (PR "Fuse the Gated
 * Delta Net inter-chunk scan into a Pallas TPU kernel", section "Changes":
 * the backward's analytic inverse gradient takes T from the forward).
 *
 * gdn_chunk_fwd_ex / gdn_chunk_bwd_ex are gdn_chunk_fwd / gdn_chunk_bwd (and,
 * with events, their timing variants) with that buffer: saved = NULL gives
 * exactly the plain calls; otherwise the forward writes w, u, P, T into it and
 * the backward reads them there, and must be given the forward's inputs
 * unchanged (q, k, v, g, beta, h0, B, T, Hk, Hv, n_segments).  Results are
 * those of the plain calls.  saved is 16-byte aligned; a smaller saved_bytes
 * than gdn_saved_bytes (for the same n_segments) gives GDN_ERR_WORKSPACE.
 * Launch order of the backward with a saved buffer: reverse walk (with
 * segments: reverse fold, reverse prefix, reverse walk), gradients.
 */
size_t gdn_saved_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments);
int gdn_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const float* h0, void* o, float* hT, int B, int T,
                     int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* saved,
                     size_t saved_bytes, void* ws, size_t ws_bytes, void* stream,
                     void* const* events, int n_events);
int gdn_chunk_bwd_ex(const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const float* h0, const void* dO, const float* dhT,
                     void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0, int B,
                     int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments,
                     const void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                     void* stream, void* const* events, int n_events);

/*
 * One GatedDeltaNet layer's use of the rule, with the element-wise operations
 * around it (PR "Shard the GatedDeltaNet sequence under
 * ici_context_parallelism", description: the layer's "qkvz" activations
 * [B, T, H, D], of which q and k enter the rule normalised and z gates its
 * output; the pages do not define these operations further, so the plain
 * forms below are this library's reading):
 *   q_n = q / sqrt(sum q^2 + 1e-6), k_n likewise, per token and key head;
 *   beta = sigmoid(b), g = -softplus(a), per token and value head -- applied
 *     by the rule's kernels where they load the gates (the logits a and b
 *     are what the caller passes);
 *   o = the rule on (q_n, k_n, v, g, beta, h0)            (as gdn_chunk_fwd);
 *   y = o * silu(z), silu(z) = z sigmoid(z)                 (z NULL: y = o).
 * The forward never forms q_n, k_n: the preparation kernel takes 1/||q|| and
 * 1/||k|| of each raw row (fp32) and applies them to its products, and the
 * walk scales its rows by them, so the unit rows are exact to fp32 rather
 * than rounded to bf16.  The backward forms bf16 copies of q_n, k_n in its
 * workspace, runs the rule's backward on them and maps dq_n, dk_n back to
 * the raw rows.
 * Forward: q, k, v, z bf16 (layouts of gdn_chunk_fwd; z as v); a, b fp32
 * [B, T, Hv]; writes y (bf16), o (bf16, the ungated output the backward needs
 * when z is given; NULL = not kept) and hT (NULL = not written).
 * Backward: the forward's inputs, o (required when z is given), the output
 * cotangent dy and dhT (NULL = 0); writes dq, dk (bf16, raw q and k, summed over
 * the value heads of each key head), dv (bf16), da, db (fp32, the logits), dz
 * (bf16, required when z is given) and dh0 (NULL = not written).
 * ws: at least gdn_layer_workspace_bytes(backward, ...) bytes; its first word
 * is the rule's status word (gdn_workspace_status).  Other conventions as for
 * gdn_chunk_fwd / gdn_chunk_bwd.
 */
size_t gdn_layer_workspace_bytes(int backward, int B, int T, int Hk, int Hv, int d_k, int d_v,
                                 int chunk, int n_segments);
int gdn_layer_fwd(const void* q, const void* k, const void* v, const float* a, const float* b,
                  const void* z, const float* h0, void* y, void* o, float* hT, int B, int T, int Hk,
                  int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws, size_t ws_bytes,
                  void* stream);
int gdn_layer_bwd(const void* q, const void* k, const void* v, const float* a, const float* b,
                  const void* z, const float* h0, const void* o, const void* dy, const float* dhT,
                  void* dq, void* dk, void* dv, float* da, float* db, void* dz, float* dh0, int B,
                  int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                  size_t ws_bytes, void* stream);

/*
 * Forward that allocates nothing and takes no workspace.  The pages have no
 * counterpart of this entry point; it exists for callers that may not
 * allocate device memory at call time and cannot lend a scratch buffer:
 * services that plan and lock all their device memory up front (where an
 * allocation could fail, fragment the plan, or stall the device while it
 * synchronises), and plug-ins whose host framework owns every byte of device
 * memory.  It computes exactly what gdn_chunk_fwd computes with
 * n_segments = 1 (same arguments otherwise, same results).
 *
 * Scratch: a fixed array inside the library's device image, sized for
 * GDN_NOALLOC_MAX_UNITS (batch x value head x chunk) units, i.e. the call
 * needs B * Hv * ceil(T / chunk) <= GDN_NOALLOC_MAX_UNITS (24 MiB of scratch);
 * larger problems are refused with GDN_ERR_WORKSPACE before anything is
 * enqueued.  Every GPU that loads the library keeps that array until the
 * process exits.
 * Set-up: a call looks up the array's device address on the current device
 * (cudaGetSymbolAddress) whenever `stream` is not capturing, and caches it per
 * device; a call made while `stream` is being captured uses that cache, so
 * make the first call on each device before any stream capture, and make one
 * again after a device reset (which reloads the library's device image at a
 * new address).
 * Sharing: all calls on a device use the same array, and its contents persist
 * from call to call.  Nothing in it needs to start at zero (each call writes
 * every scratch byte it reads before reading it), but calls whose executions
 * overlap on the GPU (different streams, or several host threads without
 * ordering) race on the array and may return wrong results: order them.
 * Never calls cudaMalloc, cudaFree or any allocating routine.
 * Failure detection: the call's kernels report a bounded wait that gave up in
 * the array's status word, which gdn_noalloc_status reads.
 */
#define GDN_NOALLOC_MAX_UNITS 256
int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const float* h0, void* o, float* hT, int B, int T,
                          int Hk, int Hv, int d_k, int d_v, int chunk, void* stream);

/*
 * Status of the bounded in-kernel waits of the last gdn_chunk_fwd_noalloc
 * call on the current device: synchronises `stream` (pass the stream that
 * call used) and reads the status word of the fixed scratch array.  Returns
 * GDN_OK if no wait gave up, GDN_ERR_TIMEOUT if one did (that call's outputs
 * are then not valid), GDN_ERR_CUDA if the stream or the read failed.  The
 * pages have no counterpart.
 */
int gdn_noalloc_status(void* stream);

/*
 * Timing variants of gdn_chunk_fwd / gdn_chunk_bwd: identical results, plus
 * cudaEventRecord(events[i], stream) right after the library's i-th kernel
 * launch, for i < n_events (NULL entries are skipped).  The events are the
 * caller's (cudaEvent_t handles created by the caller).  Launch order:
 *   forward,  n_segments = 1:  prep, walk
 *   forward,  n_segments > 1:  prep, fold, segment prefix, walk
 *   backward, n_segments = 1:  prep, walks (state recompute beside the reverse
 *                              walk, one launch), gradients
 *   backward, n_segments > 1:  prep, fold, prefix, reverse fold, reverse prefix,
 *                              walks (the two replays, one launch), gradients
 * With T == 0 or B == 0 no kernel is launched and no event is recorded.
 * Pages: none (instrumentation of the same operations).
 */
int gdn_chunk_fwd_timed(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* h0, void* o, float* hT, int B, int T,
                        int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                        size_t ws_bytes, void* stream, void* const* events, int n_events);
int gdn_chunk_bwd_timed(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* h0, const void* dO, const float* dhT,
                        void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0, int B,
                        int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments,
                        void* ws, size_t ws_bytes, void* stream, void* const* events,
                        int n_events);

/*
 * Inclusive prefix of affine maps along n, per batch row:
 *   (A_out[i], B_out[i]) = (A_i, B_i) o (A_{i-1}, B_{i-1}) o ... o (A_0, B_0)
 * with (A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2), i.e. A_out[i] h + B_out[i] is
 * h pushed through maps 0..i in order.  This is the prefix the pages take over
 * the gathered per-device pairs (PR "Shard the GatedDeltaNet sequence ...",
 * description; issue "GatedDeltaNet does not support ...", composition law).
 * A, A_out: fp32 [batch, n, d_k, d_k]; B, B_out: fp32 [batch, n, d_k, d_v];
 * row-major.  The exclusive prefix and its application to an initial state
 * are the caller's.  Sizes: d_k = 128, d_v a multiple of 16 up to 128.
 * Out-of-place only (outputs must not overlap inputs).
 */
int gdn_affine_compose(const float* A, const float* B, float* A_out, float* B_out, int batch,
                       int n, int d_k, int d_v, void* stream);

/*
 * Per-segment affine maps of the inter-chunk recurrence (pass 1 of the
 * two-pass scan, returned to the caller).  The N = ceil(T/chunk) chunks of
 * each (b, value head) are split into n_segments segments of whole chunks
 * (segment s holds chunks [floor(sN/S), floor((s+1)N/S))), and each segment's
 * chunk maps h' = A_c h + B_c, A_c = exp(g_last) I - k_g^T w, B_c = k_g^T u, are
 * composed in order: for every segment
 *     A_s = A_{last} ... A_{first},   B_s = the state the segment leaves from h = 0,
 * so the state leaving segment s is A_s h_in + B_s.  A caller that holds a
 * sequence split across devices folds each device's chunks (n_segments = 1),
 * gathers the pairs, takes the exclusive prefix (gdn_affine_compose and one
 * application to h0) and replays with gdn_chunk_fwd from its incoming state.
 * Sources: PR "Shard the GatedDeltaNet sequence under ici_context_parallelism",
 * description (each device folds its chunks into one (A, B), the pairs are
 * gathered and prefix-composed), and the A-output design question in the
 * review thread of PR "Fuse the Gated Delta Net inter-chunk scan into a
 * Pallas TPU kernel" (A as an optional output beside B).
 * A_out: fp32 [B, Hv, n_segments, d_k, d_k] (NULL = not written);
 * B_out: fp32 [B, Hv, n_segments, d_k, d_v] (required).  Row-major.
 * 1 <= n_segments <= max(1, N), else GDN_ERR_ARG.  T = 0 gives (I, 0).
 * ws: at least gdn_fwd_workspace_bytes(B, T, Hk, Hv, d_k, d_v, chunk, 1)
 * bytes, with the status word as for the forward (gdn_workspace_status).
 */
int gdn_segment_fold(const void* k, const void* v, const float* g, const float* beta,
                     float* A_out, float* B_out, int B, int T, int Hk, int Hv, int d_k, int d_v,
                     int chunk, int n_segments, void* ws, size_t ws_bytes, void* stream);

/*
 * Debug export of the per-chunk UT quantities, for tests.  For every
 * (b, value head j, chunk c), in [B, Hv, N, ...] order with N = ceil(T/chunk):
 *   S_out [.., chunk, chunk] fp32  S = tril(diag(beta) (K K^T * decay), -1)
 *   T_out [.., chunk, chunk] fp32  T = (I + S)^-1 (the device's ladder)
 *   w_out [.., chunk, d_k]   bf16  w = T diag(beta exp(G)) K
 *   u_out [.., chunk, d_v]   bf16  u = T diag(beta) V
 * Any output may be NULL.  Rows of a ragged last chunk beyond T are the
 * zero-padding rows.  Uses no workspace.  With chunk = 64 the outputs are
 * the device's 128-row tiles, N = ceil(T/128) per (b, j), each holding two
 * chunks: S_out, T_out [.., 128, 128] block diagonal (chunk 2t in rows and
 * columns 0-63 of tile t, chunk 2t + 1 in 64-127, zeros elsewhere), w_out and
 * u_out [.., 128, d] (chunk 2t in rows 0-63, chunk 2t + 1 in rows 64-127).
 */
int gdn_debug_ut(const void* k, const void* v, const float* g,
                 const float* beta, float* S_out, float* T_out, void* w_out, void* u_out,
                 int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk, void* stream);

/*
 * Status of the bounded in-kernel waits of the last gdn_chunk_fwd,
 * gdn_chunk_bwd call that used workspace `ws`.
 * The pages have no counterpart: it reports the failure detection of these
 * kernels.  Synchronises `stream` (the one exception to "never synchronises")
 * and reads the workspace's status word.  Returns GDN_OK if no wait gave up,
 * GDN_ERR_TIMEOUT if one did (the outputs of that call are then not valid),
 * GDN_ERR_ARG for a null ws, GDN_ERR_CUDA if the stream or the copy failed.
 */
int gdn_workspace_status(const void* ws, void* stream);

/*
 * Self-test of the bounded waits.  The pages have no counterpart.  Enqueues
 * one block whose wait on a barrier that nothing ever signals has to give up
 * after about limit_ns nanoseconds (1e3 <= limit_ns <= 1e10; counted in SM
 * cycles at the device's maximum clock, so longer at lower clocks); the kernel then sets
 * bit 0 of *status and returns normally (bit 1 would mean the wait completed,
 * which cannot happen), leaving the context usable.  status: one device int,
 * cleared by this call.  Synchronises `stream`.  Returns GDN_ERR_TIMEOUT when
 * the timeout was recorded (the expected outcome), GDN_OK if it was not,
 * GDN_ERR_ARG for a null status or a limit out of range, GDN_ERR_CUDA on a
 * CUDA error.
 */
int gdn_selftest_wait_timeout(long long limit_ns, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */

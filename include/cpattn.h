/*
 * cpattn.h -- C ABI of the GB300 (sm_103a) context-parallel ring-attention forward.
 *
 * The library computes, on one GPU, the forward pass of ring attention over n_cp virtual
 * context-parallel ranks: every rank's query chunk attends to every key/value block in ring
 * order with an exact online-softmax merge, under contiguous, zigzag or striped token
 * placement, with causal block skipping and grouped-query heads.
 *
 * Sources, cited by page title and section:
 *   [CEX] "Context and expert parallelism" (zerotofrontier.app): "Splitting the sequence, and
 *         the one layer that objects"; "Pass them around a ring" paragraph and the online
 *         softmax paragraph after it; "What context parallelism communicates"; "The causal
 *         mask unbalances the sequence"; "In PyTorch" (position ids sharded with the sequence).
 *   [CPC] "Context Parallelism (CP)" concept page: "Key math / How it works".
 *   [CPP] "primitive-context-parallel" skill page: "What it does"; "Interface (V1 stub)".
 *
 * Conventions for every call:
 *   - The caller owns all device memory (inputs, outputs, workspace). A plan owns only host
 *     tables and, once the ring-step path is used, two CUDA events.
 *   - Device pointers must be 16-byte aligned. bf16 tensors are raw bf16 (uint16 storage).
 *   - Calls are asynchronous on the given stream(s) and never synchronise the host, except
 *     cpattn_check, which reads the workspace's error word.
 *   - Argument errors are found on the host and returned before anything is launched; the
 *     message is available from cpattn_last_error() on the same thread.
 *   - Device-side errors (a bounded wait that ran out) are recorded in the workspace header
 *     and reported by cpattn_check. No call traps, asserts on the device or throws.
 *   - Forward calls multiply the exponentials P by V in fp16 (both tensor-core operands fp16, fp32
 *     accumulation): V is converted from bf16 during placement, exactly for 2^-14 <= |v| <= 65504
 *     (below 2^-14 within 2^-25). A V value beyond 65504, infinite or NaN makes the call compute
 *     nothing; cpattn_check (cpattn_check_noalloc) then returns CPATTN_ERR_INVALID saying so.
 *     The backward calls keep V in bf16.
 *   - There is no CPU fallback: without a usable sm_103a device, calls return CPATTN_ERR_CUDA.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Token placement of [CEX] "The causal mask unbalances the sequence":
 *   CONTIGUOUS: rank r holds tokens [r*n, (r+1)*n), n = T/n_cp ([CPP] "What it does").
 *   ZIGZAG:     2*n_cp chunks of m = T/(2 n_cp); rank r holds chunk r, then chunk 2n_cp-1-r.
 *   STRIPED:    round-robin tokens; rank r holds t = j*n_cp + r at local index j. */
typedef enum { CPATTN_CONTIGUOUS = 0, CPATTN_ZIGZAG = 1, CPATTN_STRIPED = 2 } cpattn_layout_t;

typedef enum {
    CPATTN_OK = 0,
    CPATTN_ERR_INVALID = 1,     /* bad argument (null pointer, shape, alignment, step order) */
    CPATTN_ERR_UNSUPPORTED = 2, /* valid but not built here (d_k not 64 or 128, ...) */
    CPATTN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    CPATTN_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has the CUDA error) */
    CPATTN_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out (from cpattn_check) */
} cpattn_status_t;

/* Block classes of [CEX] "The causal mask unbalances the sequence". */
typedef enum { CPATTN_TILE_FULL = 0, CPATTN_TILE_DIAG = 1, CPATTN_TILE_SKIP = 2 } cpattn_tile_class_t;

typedef struct cpattn_plan* cpattn_plan_t;   /* opaque, host-side */
typedef struct CUstream_st* cpattn_stream_t; /* a cudaStream_t; NULL is the legacy default stream */

/* Build a plan for T tokens, h query heads, n_kv key/value heads (h % n_kv == 0; query head i
 * reads KV head i / (h/n_kv)), head width d_k (64 or 128), n_cp virtual ranks, a layout and a
 * causal flag. Requires T % n_cp == 0 (ZIGZAG: T % (2 n_cp) == 0). The plan computes, for the
 * default positions 0..T-1, the block class of every (rank, ring step, query tile, key tile),
 * the per-rank work and byte counters and a longest-first order of the query tiles. Host only;
 * no CUDA call. *out is set on success. */
cpattn_status_t cpattn_plan(int64_t T, int h, int n_kv, int d_k, int n_cp, cpattn_layout_t layout, int causal,
                            cpattn_plan_t* out);
cpattn_status_t cpattn_plan_destroy(cpattn_plan_t plan);

/* The attention kernel is persistent: one CTA per SM holds the SM's whole register file until the
 * work runs out, so work on other streams that needs SMs (a device-to-device copy of the ring's
 * next block, a communication library's transfer kernel) waits for the launch's tail. With sms > 0
 * the plan's forward attention launches leave that many SMs free, so such transfers can run beside
 * the step they must precede ([CEX] "When the ring hides its communication"). Default 0; a value
 * at or above the device's SM count leaves one CTA. Host only. */
cpattn_status_t cpattn_plan_set_reserved_sms(cpattn_plan_t plan, int sms);

/* Workspace bytes for cpattn_forward / cpattn_permute with batch B. */
cpattn_status_t cpattn_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);
/* Workspace bytes for the ring-step path (permute + ring_step + finalize): the forward
 * workspace plus the two-slot key/value stage and the fp32 running state (O unnormalised against
 * a running maximum, with the running sum). */
cpattn_status_t cpattn_ring_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);

/* The whole forward pass ([CEX] "Pass them around a ring" and the online-softmax paragraph;
 * [CPC] "Key math / How it works"): place tokens, run every virtual rank over every ring step
 * with causal block skipping, normalise and write the result back in natural token order.
 *   q   [B, T, h, d_k]    bf16, natural token order          (device, read)
 *   k,v [B, T, n_kv, d_k] bf16, natural token order          (device, read)
 *   pos [T] int32 position id of each natural token, or NULL for 0..T-1 (device, read). The
 *       causal mask shows key u to query t iff pos[u] <= pos[t]; positions travel with the
 *       tokens ([CEX] "In PyTorch").
 *   scale: softmax scale; <= 0 means 1/sqrt(d_k).
 *   o   [B, T, h, d_k] bf16 output, natural order            (device, written)
 *   lse [B, h, T] fp32 natural-log log-sum-exp of the scaled visible scores (device, written;
 *       -inf for a row that sees no key, whose o row is then 0)
 *   ws, ws_bytes: workspace of at least cpattn_workspace_size bytes (device, scratch).
 * Enqueued on `stream`. */
cpattn_status_t cpattn_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                               const int32_t* pos, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                               cpattn_stream_t stream);

/* cpattn_forward without the placement step: every virtual rank over every ring step on a
 * workspace that cpattn_permute has filled, writing o and lse as cpattn_forward does. Lets a
 * caller place tokens once and run the attention (or time the two kernels) separately. */
cpattn_status_t cpattn_attend(cpattn_plan_t plan, int B, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                              cpattn_stream_t stream);

/* cpattn_forward for callers that cannot allocate device memory. The source pages describe no
 * such call: it exists for code that may not call cudaMalloc or any other allocating routine,
 * such as code running inside a memory allocator's own hooks (where allocating again would
 * recurse), a plug-in loaded into a host process that owns every device memory pool, or a
 * real-time loop that may not wait on an allocation.
 * Same arguments as cpattn_forward minus the workspace: the scratch is a 64 MiB device array
 * built into the library, which every GPU that loads the library holds until the process
 * exits. The call allocates nothing, on the device or on the host (the unit order reaches the
 * device inside kernel parameters). A problem whose cpattn_workspace_size exceeds 64 MiB is
 * rejected with CPATTN_ERR_WORKSPACE and a message saying so.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before capturing a stream.
 *   - All calls share the array and it keeps the last call's contents; each call clears what
 *     must start at zero. Calls that overlap on the GPU (other streams, other threads) race on
 *     it: issue them one after another on one stream.
 *   - A device-side timeout is recorded in the array's header: after synchronising the stream,
 *     cpattn_check_noalloc reports it as cpattn_check does for a caller-owned workspace. */
cpattn_status_t cpattn_forward_noalloc(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const int32_t* pos, float scale, void* o, float* lse,
                                       cpattn_stream_t stream);
/* cpattn_check for the built-in scratch of cpattn_forward_noalloc on the current device: after
 * the stream has been synchronised, CPATTN_OK or CPATTN_ERR_TIMEOUT (the message names the wait).
 * Allocates nothing. */
cpattn_status_t cpattn_check_noalloc(cpattn_plan_t plan);
/* cpattn_selftest_wait_timeout on the built-in scratch of the current device: records a timeout
 * there exactly as a kernel wait that ran out would, so that cpattn_check_noalloc can be tested.
 * The next cpattn_forward_noalloc clears it. */
cpattn_status_t cpattn_selftest_wait_timeout_noalloc(uint64_t timeout_ns, cpattn_stream_t stream);

/* Ring-faithful path, step 1: gather Q, K, V and the position ids into layout order inside the
 * workspace (rank-major blocks) and reset the workspace header. Same arguments as
 * cpattn_forward's inputs; ws must hold cpattn_ring_workspace_size bytes to be usable by
 * cpattn_ring_step (cpattn_workspace_size is enough for the permute alone). */
cpattn_status_t cpattn_permute(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                               const int32_t* pos, void* ws, size_t ws_bytes, cpattn_stream_t stream);

/* Ring-faithful path, step 2 ([CEX] "Pass them around a ring"): ring step `step` of n_cp for
 * every virtual rank at once. Rank r attends to the key/value block it holds, that of rank
 * (r - step) mod n_cp, read from the stage slot step % 2 (step 0: its own block in place), and
 * merges the partial (O_s with its maximum and sum) into the fp32 running state in the workspace
 * (the online-softmax merge; cpattn_finalize normalises). It also performs the hop to the next
 * step: every rank's slot (step+1) % 2 receives the block its left neighbour holds now (send
 * right, receive left). With `copy` NULL the step's own kernel does it: its otherwise idle warps
 * copy the blocks while the attention runs, so the hop ends with the step and everything stays
 * on `compute`. With a `copy` stream the hop is enqueued there as device-to-device copies,
 * ordered against the compute stream with events so that a slot is overwritten only after the
 * step that read it has finished. One pass uses one kind of hop at every step. Steps must be
 * issued in order 0..n_cp-1 after cpattn_permute, from one host thread per plan, with
 * cpattn_permute and cpattn_finalize on the stream passed here as `compute` (step 0 orders the
 * copy stream after the compute stream only), and with the B cpattn_permute placed; otherwise
 * CPATTN_ERR_INVALID before any launch. */
cpattn_status_t cpattn_ring_step(cpattn_plan_t plan, int B, int step, float scale, void* ws, size_t ws_bytes,
                                 cpattn_stream_t compute, cpattn_stream_t copy);

/* Ring-faithful path, step 3: the running state after the last step, normalised, rounded to
 * bf16 and written back in natural token order: o [B,T,h,d_k] bf16, lse [B,h,T] fp32. */
cpattn_status_t cpattn_finalize(cpattn_plan_t plan, int B, void* o, float* lse, void* ws, size_t ws_bytes,
                                cpattn_stream_t stream);

/* The forward under a per-query lower bound on the visible key positions: key u is visible to
 * query t iff lo[t] <= pos[u] <= pos[t]. With positions 0..T-1 (pos NULL) and lo[t] = the first
 * token of t's document this is the document mask of packed sequences ([CEX] "What context
 * parallelism communicates": the all-gather variant "makes arbitrary masks, such as document
 * masks for packed sequences, easy to support"; on one GPU every rank's queries already read the
 * resident keys and values of all ranks, which is that variant's data flow). Masks on positions
 * only, so the mask positions must increase through the packed sequence; per-document position
 * ids (for rotary embeddings) are not what pos means here.
 *   lo [T] int32 (device, natural order, 16-byte aligned); the plan must be causal, else
 *   CPATTN_ERR_UNSUPPORTED. Other arguments as cpattn_forward. A row that sees no key gets
 *   o = 0 and lse = -inf. */
cpattn_status_t cpattn_forward_masked(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                      const int32_t* pos, const int32_t* lo, float scale, void* o, float* lse, void* ws,
                                      size_t ws_bytes, cpattn_stream_t stream);

/* The forward under document ids ([CEX] "What context parallelism communicates": masks "such as
 * document masks for packed sequences"): key u is visible to query t iff doc[u] == doc[t] and, for
 * a causal plan, pos[u] <= pos[t]. Any int32 ids in any order; a document need not be contiguous.
 * The ids travel with the tokens; each tile's (min, max) id, with the position ranges, classifies
 * every (query tile, key tile) pair, and the key tiles some query of a row group may see are
 * recorded per ring step as a bitmask the kernel's walkers follow. A row that sees no key gets
 * o = 0 and lse = -inf.
 *   doc [T] int32 (device, natural order, 16-byte aligned); other arguments as cpattn_forward. */
cpattn_status_t cpattn_forward_docs(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                    const int32_t* pos, const int32_t* doc, float scale, void* o, float* lse, void* ws,
                                    size_t ws_bytes, cpattn_stream_t stream);

/* Backward pass ([CEX] "What context parallelism communicates": each rank keeps the gradient
 * of its own queries; the key and value gradients travel back to their owners as a second
 * circulating block of the ring, which on one GPU is a key tile's gradient accumulated over
 * every rank's queries in ring order). For the loss L = sum <O, dO>:
 *   P = exp(scale q.k - lse), D_t = <dO_t, O_t>, dS = P (<dO_t, v_u> - D_t),
 *   dq = scale sum_u dS k_u,  dk = scale sum_t dS q_t,  dv = sum_t P dO_t
 * (dk, dv summed over the query heads of each KV group).
 *   q, k, v, pos, scale   as passed to cpattn_forward (natural order, device)
 *   o [B,T,h,d_k] bf16, lse [B,h,T] fp32   the forward's outputs (device, read)
 *   dout [B,T,h,d_k] bf16                  gradient of the loss w.r.t. o (device, read)
 *   dq [B,T,h,d_k], dk, dv [B,T,n_kv,d_k]  bf16 gradients, natural order (device, written)
 *   ws / ws_bytes  at least cpattn_backward_workspace_size(plan, B) bytes, 1024-byte aligned.
 * Every pointer non-NULL and 16-byte aligned (pos may be NULL), or CPATTN_ERR_INVALID before any
 * launch. Asynchronous on `stream`; device-side timeouts are read by cpattn_check. */
/* Bytes each rank receives in one backward pass of the ring ([CEX] "What context parallelism
 * communicates": the key/value gradients travel back to their owners as a second circulating
 * block, roughly doubling the traffic): the other n_cp - 1 ranks' K and V blocks in bf16, and the
 * n_cp arrivals of the circulating dK and dV blocks as fp32 partial sums (the last hop returns a
 * rank's own block): 4 B n d_kv (n_cp - 1) + 8 B n d_kv n_cp. bytes_recv [n_cp] (host, written).
 * Host only. The fused backward keeps each block's partial sums in tensor memory; the ring-step
 * backward (cpattn_backward_ring_step) moves exactly these bytes between the ranks' slots. */
cpattn_status_t cpattn_backward_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv);
cpattn_status_t cpattn_backward_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);
cpattn_status_t cpattn_backward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, const int32_t* pos, float scale, void* dq, void* dk,
                                void* dv, void* ws, size_t ws_bytes, cpattn_stream_t stream);

/* The backward pass under the per-query lower bound of cpattn_forward_masked (document masks of
 * packed sequences: "the backward pass is the mirror image", [CEX] "What context parallelism
 * communicates"). lo [T] int32 as for cpattn_forward_masked; the plan must be causal, else
 * CPATTN_ERR_UNSUPPORTED. Other arguments as cpattn_backward. */
cpattn_status_t cpattn_backward_masked(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const void* o, const float* lse, const void* dout, const int32_t* pos,
                                       const int32_t* lo, float scale, void* dq, void* dk, void* dv, void* ws,
                                       size_t ws_bytes, cpattn_stream_t stream);

/* The backward pass as ring steps ([CEX] "What context parallelism communicates": each rank
 * keeps the gradient of its own queries; the key and value gradients of a block travel with the
 * block as a second circulating block and return to its owner). Same result as cpattn_backward
 * (without document masks), computed step by step with the ring's data movement made explicit:
 *   cpattn_backward_begin: placement and the backward's side data (arguments as
 *     cpattn_backward's inputs). ws / ws_bytes at least cpattn_backward_ring_workspace_size(plan,
 *     B) bytes, 1024-byte aligned.
 *   cpattn_backward_ring_step, steps 0..n_cp-1 in order, from one host thread per plan: on
 *     `compute`, every rank r computes, against its own queries, the dK/dV contribution for the
 *     block it holds (that of rank (r - step) mod n_cp; step 0 its own) and adds its dQ for that
 *     block into its running fp32 dQ; the contribution is added into the block's fp32 partial
 *     sum, which arrived with the block (the dQ work runs first, while that sum is in flight).
 *     On `copy`: the K/V hop for the next step (issued first, overlapping this step's kernels)
 *     and the hop of the partial sums to the right neighbour;
 *     after the last step that hop returns each block's sums to its owner. Events order the two
 *     streams so that no slot is overwritten before the step that read it has finished.
 *   cpattn_backward_finalize: once the returning sums have arrived, dq [B,T,h,d_k] and dk, dv
 *     [B,T,n_kv,d_k] bf16 in natural order (device, written, 16-byte aligned), on `stream`.
 * cpattn_backward_begin and cpattn_backward_finalize must run on the stream passed to the steps
 * as `compute` (step 0 orders the copy stream after the compute stream only). Out-of-order steps,
 * a B other than cpattn_backward_begin's, or a finalize before the last step return
 * CPATTN_ERR_INVALID before any launch. Asynchronous; device-side timeouts are read by
 * cpattn_check(plan, ws). */
cpattn_status_t cpattn_backward_ring_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);
cpattn_status_t cpattn_backward_begin(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout, const int32_t* pos, void* ws,
                                      size_t ws_bytes, cpattn_stream_t stream);
cpattn_status_t cpattn_backward_ring_step(cpattn_plan_t plan, int B, int step, float scale, void* ws, size_t ws_bytes,
                                          cpattn_stream_t compute, cpattn_stream_t copy);
cpattn_status_t cpattn_backward_finalize(cpattn_plan_t plan, int B, void* dq, void* dk, void* dv, void* ws,
                                         size_t ws_bytes, cpattn_stream_t stream);

/* Ulysses, the head split ([CEX] "Ulysses, splitting by heads instead"), as a comparison
 * workload on one GPU with n_cp virtual ranks. Rank r starts with the tokens r n .. r n + n - 1
 * (n = T / n_cp) of every head; a first all-to-all gives every rank all T tokens of its
 * hp = h / n_cp query heads r hp .. r hp + hp - 1 and of the KV heads they use; each rank runs
 * exact attention on them; a second all-to-all returns the outputs to the token split. The KV
 * heads of a rank are (r hp) / g + j for j < n_kv / n_cp (g = h / n_kv). When n_cp > n_kv each
 * rank holds the one KV head its query heads use, replicated on n_cp / n_kv ranks.
 *   cpattn_ulysses_plan: h a multiple of n_cp (whole heads per rank); n_cp a divisor or a
 *   multiple of n_kv; T a multiple of n_cp; d_k 64 or 128; else CPATTN_ERR_INVALID /
 *   CPATTN_ERR_UNSUPPORTED. The plan works only with the cpattn_ulysses_* calls (the other
 *   calls return CPATTN_ERR_INVALID for it) and is destroyed by cpattn_plan_destroy.
 *   cpattn_ulysses_counts: bytes_recv [n_cp] (host, written), the bytes rank r receives in the
 *   two all-to-alls of one forward pass for B sequences: the other ranks' n tokens of its query
 *   heads, its KV heads (K and V) and, back, of the other ranks' output heads for its own tokens,
 *   2 bytes a number: 2 B n d_k (n_cp - 1) (2 hp + 2 nkv_r) with nkv_r its KV heads.
 *   cpattn_ulysses_forward: arguments, layouts and results as cpattn_forward (natural order,
 *   device pointers, 16-byte aligned; pos NULL or T int32 positions), the workspace at least
 *   cpattn_ulysses_workspace_size(plan, B) bytes, 1024-byte aligned. The result equals plain
 *   attention (head split changes no arithmetic of a head). Asynchronous on `stream`;
 *   device-side timeouts are read by cpattn_check(plan, ws). */
cpattn_status_t cpattn_ulysses_plan(int64_t T, int h, int n_kv, int d_k, int n_cp, int causal, cpattn_plan_t* out);
cpattn_status_t cpattn_ulysses_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);
cpattn_status_t cpattn_ulysses_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv);
cpattn_status_t cpattn_ulysses_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const int32_t* pos, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                                       cpattn_stream_t stream);

/* The all-gather variant ([CEX] "Splitting the sequence, and the one layer that objects": gather
 * the keys and values so that every rank holds the full K and V, then compute attention for the
 * local queries; [CEX] "What context parallelism communicates": the all-gather moves every block
 * before the attention kernel runs, so its time is exposed, and it works with one ordinary
 * attention kernel). On one GPU every virtual rank r gets its own gathered copy of the whole K and
 * V (rank-major layout order; [n_cp][n_cp][B][n_kv][n][d_k] bf16 in the workspace) by device-to-
 * device copies, and one attention launch then computes every rank's queries, each rank reading
 * only its own copy. The result equals cpattn_forward's (same arithmetic in the same order).
 *   cpattn_allgather_workspace_size: the forward workspace plus the gathered copies
 *     (2 n_cp times the bf16 K and V of the batch).
 *   cpattn_allgather_forward: placement, the gather, the attention; arguments as
 *     cpattn_forward_masked with lo optional (NULL: causal or non-causal as the plan says; else the
 *     per-query lower bound of cpattn_forward_masked, which needs a causal plan).
 *   cpattn_allgather_gather / cpattn_allgather_attend: the last two phases alone, on a workspace
 *     cpattn_permute has filled (lets a caller time the exposed gather beside the attention).
 *   cpattn_allgather_counts: bytes_recv [n_cp] (host, written), the bytes rank r receives in the
 *     gather: the other n_cp - 1 ranks' K and V blocks, 4 B n d_kv (n_cp - 1) with d_kv = n_kv d_k,
 *     the same volume as the ring ([CEX] "What context parallelism communicates": "Both come to").
 * Device pointers 16-byte aligned, the workspace 1024-byte aligned; asynchronous on `stream`;
 * device-side timeouts are read by cpattn_check(plan, ws). */
cpattn_status_t cpattn_allgather_workspace_size(cpattn_plan_t plan, int B, size_t* bytes);
cpattn_status_t cpattn_allgather_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv);
cpattn_status_t cpattn_allgather_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                         const int32_t* pos, const int32_t* lo, float scale, void* o, float* lse,
                                         void* ws, size_t ws_bytes, cpattn_stream_t stream);
/* cpattn_allgather_forward under document ids (as cpattn_forward_docs): any ids, in any order. */
cpattn_status_t cpattn_allgather_forward_docs(cpattn_plan_t plan, int B, const void* q, const void* k,
                                              const void* v, const int32_t* pos, const int32_t* doc, float scale,
                                              void* o, float* lse, void* ws, size_t ws_bytes, cpattn_stream_t stream);
cpattn_status_t cpattn_allgather_gather(cpattn_plan_t plan, int B, void* ws, size_t ws_bytes, cpattn_stream_t stream);
cpattn_status_t cpattn_allgather_attend(cpattn_plan_t plan, int B, float scale, void* o, float* lse, void* ws,
                                        size_t ws_bytes, cpattn_stream_t stream);

/* One process of a ring that spans processes (one process per GPU; [CEX] "Pass them around a
 * ring": each rank computes its queries against the key/value block it holds while it sends that
 * block to its right neighbour and receives the next from its left; "When the ring hides its
 * communication": each transfer overlaps a step of attention). A process holds the R consecutive
 * ranks rank0 .. rank0 + R - 1 of the plan's n_cp (R = n_cp: the whole ring in one process). The
 * library computes and moves blocks between the process's own ranks; the caller moves the one
 * block per step that crosses to the next process (rank rank0 + R - 1 -> rank rank0 + R) with its
 * own transport (NCCL send/receive, peer copies, or host memory), into the next process's slot.
 *   Stage slot (device, caller-owned, 1024-byte aligned, two of them for the double buffer): the
 *     blocks the R ranks hold, in four regions: K and V [R][B][n_kv][n][d_k] bf16, the blocks'
 *     position ids [R][n] int32 and their tile table [R][n_qt] int32x4 (positions travel with the
 *     block: [CEX] "In PyTorch"). Region x starts at region_offset[x] of the slot and local rank
 *     i's block in it at region_offset[x] + i block_bytes[x] (x = K, V, positions, tiles).
 *   cpattn_dist_sizes: the workspace bytes, slot bytes and the four regions' offsets and block
 *     bytes (host, written; any pointer may be NULL).
 *   cpattn_dist_begin: q [B][R n][h][d_k], k, v [B][R n][n_kv][d_k] bf16 (device): the process's
 *     tokens, rank rank0's n tokens in its local layout order, then rank rank0 + 1's, ...; pos
 *     [R n] int32 position ids of those tokens or NULL for their natural positions under the
 *     plan's layout; lo [R n] int32 or NULL: the per-query lower bound of cpattn_forward_masked
 *     (document masks; a causal plan), which stays with the queries while the keys' positions
 *     travel. Places the queries in the workspace and the own blocks in `slot`.
 *   cpattn_dist_step, steps 0..n_cp-1 in order from one host thread: every local rank attends to
 *     the block it holds in `slot` (at step s, that of rank (r - s) mod n_cp) and merges the result
 *     into its fp32 running state in the workspace. The slot must not change until the step's
 *     work on `stream` has finished.
 *   cpattn_dist_shift: on `stream`, local rank i + 1's block in dst_slot <- local rank i's block
 *     in src_slot, for i < R - 1, all four regions; with wrap != 0 (a process that holds the whole
 *     ring) also local rank 0's block <- local rank R - 1's. Otherwise local rank 0's block in
 *     dst_slot is the caller's to fill with the block the previous process sends.
 *   cpattn_dist_step_shift: cpattn_dist_step on `slot` and cpattn_dist_shift from `slot` into
 *     next_slot (a different slot) on the same stream, in one call: the K and V blocks move inside
 *     the step's kernel, by warps that have no part in the attention, while it runs; the position
 *     tables follow by copies on `stream`. next_slot must not be read by anyone until the call's
 *     work on `stream` has finished; it must not be written either, except local rank 0's block
 *     when wrap is 0 (the transport's).
 *   cpattn_dist_finalize: after the last step, o [B][R n][h][d_k] bf16 and lse [B][h][R n] fp32 in
 *     the process's token order (that of q).
 * Out-of-order steps, or a B, rank0 or R other than cpattn_dist_begin's, return CPATTN_ERR_INVALID
 * before any launch. Device-side timeouts are recorded in the workspace header (cpattn_check). */
cpattn_status_t cpattn_dist_sizes(cpattn_plan_t plan, int B, int R, size_t* ws_bytes, size_t* slot_bytes,
                                  size_t* region_offset /* [4] */, size_t* block_bytes /* [4] */);
cpattn_status_t cpattn_dist_begin(cpattn_plan_t plan, int B, int rank0, int R, const void* q, const void* k,
                                  const void* v, const int32_t* pos, const int32_t* lo, void* ws, size_t ws_bytes,
                                  void* slot, size_t slot_bytes, cpattn_stream_t stream);
cpattn_status_t cpattn_dist_step(cpattn_plan_t plan, int B, int rank0, int R, int step, float scale,
                                 const void* slot, size_t slot_bytes, void* ws, size_t ws_bytes,
                                 cpattn_stream_t stream);
cpattn_status_t cpattn_dist_shift(cpattn_plan_t plan, int B, int R, const void* src_slot, void* dst_slot,
                                  size_t slot_bytes, int wrap, cpattn_stream_t stream);
cpattn_status_t cpattn_dist_step_shift(cpattn_plan_t plan, int B, int rank0, int R, int step, float scale,
                                       const void* slot, void* next_slot, int wrap, size_t slot_bytes, void* ws,
                                       size_t ws_bytes, cpattn_stream_t stream);
cpattn_status_t cpattn_dist_finalize(cpattn_plan_t plan, int B, int rank0, int R, void* o, float* lse, void* ws,
                                     size_t ws_bytes, cpattn_stream_t stream);

/* S-way log-sum-exp merge of partial attention results ([CEX] online-softmax paragraph: old
 * totals rescaled to a common maximum). For every row and head:
 *   lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) * o_s;  all lse_s = -inf gives (0, -inf).
 *   o_parts   [S][rows][h][d] fp32 (device, read)      lse_parts [S][h][rows] fp32 (device, read)
 *   o_bf16    [rows][h][d] bf16 (device, written)      lse       [h][rows] fp32 (device, written)
 * d must be a multiple of 8 (each thread of the kernel merges 8 consecutive values). */
cpattn_status_t cpattn_merge(int S, int64_t rows, int h, int d, const float* o_parts, const float* lse_parts,
                             void* o_bf16, float* lse, cpattn_stream_t stream);

/* The plan's block decisions and work counters (host memory, written by the call):
 *   tiles_full/diag/skip [n_cp * n_cp], index r * n_cp + step: tile counts of one (batch
 *       element, query head) for rank r at ring step `step`, tiles of block_q x block_k tokens
 *       over each rank's local order (the last tile of a block may be short);
 *   pairs [n_cp]: exact visible (query, key) pairs of rank r for one (batch element, head);
 *   kv_bytes_recv [n_cp]: bytes of K and V rank r receives around the ring for the batch:
 *       4 * B * n * n_kv * d_k * (n_cp - 1) ([CEX] "What context parallelism communicates");
 *   half_units [n_cp]: chunk-level work, FULL chunk pairs count 2 and partly visible ones 1
 *       ([CEX] "The causal mask unbalances the sequence").
 * Any output pointer may be NULL. Positions are 0..T-1. */
cpattn_status_t cpattn_plan_counts(cpattn_plan_t plan, int B, int64_t* tiles_full, int64_t* tiles_diag,
                                   int64_t* tiles_skip, int64_t* pairs, int64_t* kv_bytes_recv,
                                   int64_t* half_units);

/* After the stream has been synchronised: the key tiles the kernels actually computed since the
 * last cpattn_forward / cpattn_permute on this workspace, summed over batch elements and query
 * heads, by (rank r, ring step): full[r * n_cp + step] tiles computed without a mask (every
 * pair visible) and diag[r * n_cp + step] partly visible tiles computed with the element mask.
 * Skipped tiles are not computed. With positions 0..T-1 these equal B * h times the plan's
 * tiles_full and tiles_diag. Host arrays of n_cp * n_cp; either may be NULL. */
cpattn_status_t cpattn_tile_counts(cpattn_plan_t plan, int B, const void* ws, int64_t* full, int64_t* diag);

/* Query and key tile sizes the plan classifies and the kernels compute with. */
cpattn_status_t cpattn_tile_shape(cpattn_plan_t plan, int* block_q, int* block_k);

/* After the stream that ran the calls has been synchronised: reads the workspace header and
 * returns CPATTN_OK, or CPATTN_ERR_TIMEOUT if a device-side wait ran out (the message names the
 * wait). ws is the device workspace. */
cpattn_status_t cpattn_check(cpattn_plan_t plan, const void* ws);

/* Failure-detection self test: launches one block that waits on a barrier nothing completes,
 * with a limit of timeout_ns nanoseconds, and records the timeout in the workspace header
 * exactly as the attention kernels do. cpattn_check then reports CPATTN_ERR_TIMEOUT. */
cpattn_status_t cpattn_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns,
                                             cpattn_stream_t stream);

/* Thread-local message of the last failed call on this thread ("" if none). */
const char* cpattn_last_error(void);

/* Library version, e.g. "cpattn 0.1 sm_103a". */
const char* cpattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */

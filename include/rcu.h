/*
 * rcu.h — C ABI of the GB300 recurrent-cell unroll library (librcu.so).
 *
 * The library runs the time-unrolled forward pass of stacked LSTM, GRU and
 * LSTM-with-projection (LSTMP) networks, padded or variable-length, and the
 * RSSM prior unroll, entirely in its own CUDA kernels (sm_103a).  The caller
 * supplies device memory and a CUDA stream; nothing here depends on PyTorch.
 *
 * Conventions shared by every entry point
 *  - Return value: RCU_OK (0) or a negative RCU_ERR_* code.  The message of
 *    the last failure on the calling host thread is returned by
 *    rcu_last_error().
 *  - Pointers named as "device" must point to memory the current CUDA device
 *    can access; all tensors are dense, row-major (C order) and fp32 unless
 *    stated.  Input and output buffers must not overlap.
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; errors detected on the
 *    device are reported by rnn_get_status / rssm_get_status.
 *  - A handle is used from one stream at a time; different handles are
 *    independent (no global mutable state, cf. the thread-local recurrent
 *    mode of "[Performance] LSTM/GRU scan: canonical strides + cuDNN
 *    flat-storage clones + thread-local recurrent mode", pytorch/rl PR 3754).
 *  - Memory ownership: the caller owns every input/output buffer.  A handle
 *    owns a private copy of its weights (made by the set_weights calls, so the
 *    caller may free or reuse its weight tensors at once; cf. the flat-storage
 *    aliasing fix in pytorch/rl PR 3754) and a workspace that grows on demand
 *    inside the forward call.
 */
#ifndef RCU_H
#define RCU_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RCU_API __attribute__((visibility("default")))
#else
#define RCU_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rcu_rnn_s *rcu_rnn_t;
typedef struct rcu_rssm_s *rcu_rssm_t;

/* Cell kinds; RCU_BIDIR may be OR-ed into the cell argument of rnn_create. */
#define RCU_LSTM 0
#define RCU_GRU 1
#define RCU_BIDIR 0x100

/* Weight storage types.  RCU_BF16: weights rounded to bf16 (nearest-even),
 * GEMM operands (x, inter-layer outputs, recurrent h, projection input m)
 * rounded to bf16; accumulation, biases, cell state and all elementwise math
 * in fp32 (the AMP-style reduced-precision LSTM discussed in "Integrating
 * CuDNN API for LSTMs with projections", pytorch/pytorch issue 46213). */
#define RCU_F32 0
#define RCU_BF16 1

/* Status codes. */
#define RCU_OK 0
#define RCU_ERR_INVALID (-1)     /* bad argument: NULL, shape, dims, layer index */
#define RCU_ERR_UNSUPPORTED (-2) /* e.g. GRU with projection; plan does not fit the GPU */
#define RCU_ERR_CUDA (-3)        /* CUDA launch or allocation failure */
#define RCU_ERR_TIMEOUT (-4)     /* a device-side step barrier gave up waiting */
#define RCU_ERR_LENGTHS (-5)     /* device found a length outside [1, T] */
#define RCU_ERR_STATE (-6)       /* weights not set for every layer/direction */

/* Attributes for rnn_set_attr / rssm_set_attr. */
#define RCU_ATTR_BARRIER_TIMEOUT_NS 1 /* bound on any device wait (default 2e9 ns) */
#define RCU_ATTR_TEST_DROP_ARRIVAL 2  /* testing only: 1 = one CTA of the forward's first
                                         recurrent kernel never arrives at the first step
                                         barrier, 2 = the same in the backward recurrence
                                         (rnn_backward); on an RSSM handle, nonzero = one CTA
                                         skips its first state broadcast.  The waits must
                                         time out (RCU_ERR_TIMEOUT from *_get_status). */
#define RCU_ATTR_FORCE_PATH 3         /* 0 = automatic, 1 = portable SIMT kernels only,
                                         2 = tensor-core (tcgen05) kernels where supported
                                         (on an fp32 handle: its GEMMs as fp32-accurate
                                         three-term bf16 splits at any size; automatic
                                         mode takes them for large products only),
                                         3 = cluster-resident recurrent kernel where W_hh
                                         fits one thread-block cluster (else SIMT).  On an
                                         RSSM handle: 0 = automatic, 1 = the backward's
                                         reverse-time chain as separate launches per step
                                         instead of one cluster-resident kernel */
#define RCU_ATTR_TRACE 5              /* 1 = record per-step timestamps (rnn_get_trace);
                                         2 = also every CTA's stamps of the tensor-core
                                         recurrence for a window of steps */
#define RCU_ATTR_TC_KSPLIT 7          /* tensor-core recurrent kernel: CTAs that split the
                                         K (= hidden) dimension of h W_hh^T, exchanging
                                         partial sums through distributed shared memory
                                         (0 = automatic: 2 where it fits, 1 = no split,
                                         2 = CTA pairs, 4 = clusters of 4; a split that
                                         does not fit falls back to the next smaller) */
#define RCU_ATTR_LAYER_PIPELINE 10    /* 1 (default) = a stacked unidirectional bf16 LSTMP
                                         whose tensor-core recurrence leaves room for a second
                                         one runs its layers concurrently over chunks of
                                         steps (layer l+1 on chunk c while layer l runs chunk
                                         c+1), on streams the handle owns; results equal the
                                         layer-by-layer ones.  0 = layer by layer */
#define RCU_ATTR_PROFILE 4            /* 1 = record a CUDA event pair around every kernel
                                         this handle launches (RSSM handle: around each
                                         named phase of launches), on the launching
                                         stream; read the totals with rnn_profile_entry /
                                         rssm_profile_entry */
#define RCU_ATTR_HOST_CHUNKS 8        /* rnn_forward_host: chunks of steps whose host<->device
                                         copies overlap the other chunks' compute (0 =
                                         automatic, 1 = none, up to RCU_MAX_HOST_CHUNKS;
                                         unidirectional networks without projection or
                                         lengths, x and y page-locked) */
#define RCU_MAX_HOST_CHUNKS 16

/* Clipping targets for rnn_set_clip. */
#define RCU_CLIP_CELL 0 /* LSTM cell state c_t */
#define RCU_CLIP_PROJ 1 /* projected hidden state h_t = W_hr m_t (LSTMP) */

/* Message of the last failure on this host thread ("" if none). */
RCU_API const char *rcu_last_error(void);

/* Library version string. */
RCU_API const char *rcu_version(void);

/* ------------------------------------------------------------------------ */
/* Stacked LSTM / GRU / LSTMP                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Create a network description.
 *   cell    RCU_LSTM or RCU_GRU, optionally | RCU_BIDIR (two directions per layer).
 *   layers  >= 1.  Layer l > 0 takes the previous layer's output (forward and
 *           backward halves concatenated).
 *   in_dim  input width of layer 0 (>= 1).
 *   hidden  H, units per direction (>= 1).
 *   proj    0 = no projection; 0 < proj < hidden = LSTMP with
 *           h_t = W_hr (o_t * tanh(c_t)) (Sak et al., the cuDNN projection
 *           named in pytorch/pytorch issue 46213).  proj > 0 with RCU_GRU is
 *           RCU_ERR_UNSUPPORTED, as the issue asks for RNN/GRU.
 *   dtype   RCU_F32 or RCU_BF16.
 * On success *out receives the handle.
 */
RCU_API int rnn_create(rcu_rnn_t *out, int cell, int layers, int in_dim, int hidden, int proj, int dtype);

/*
 * Copy one layer/direction's weights into the handle (PyTorch nn.LSTM/nn.GRU
 * layout, device pointers, fp32).  Gate row order: LSTM i,f,g,o; GRU r,z,n.
 *   W_ih [nG*H, in_l]  in_l = in_dim for layer 0, D*Hout after (Hout = proj or H)
 *   W_hh [nG*H, Hout]
 *   b_ih, b_hh [nG*H]  NULL means zero ("with and without bias",
 *                      pytorch/pytorch issue 46213)
 *   W_hr [proj, H]     required iff proj > 0, else must be NULL
 * dir is 0, or 1 for the backward direction of a bidirectional network.
 * The copy is ordered on `stream`; the caller may reuse its buffers once the
 * stream has passed this call.
 */
RCU_API int rnn_set_weights(rcu_rnn_t h, int layer, int dir, const float *W_ih, const float *W_hh,
                    const float *b_ih, const float *b_hh, const float *W_hr, void *stream);

/*
 * Forward pass over T steps of B sequences (time-major).
 *   x        [T, B, in_dim] device.
 *   lengths  NULL (every row has length T) or device int32 [B] with
 *            1 <= lengths[b] <= T.  Rows are sorted by length on the device
 *            and packed (pack/unpack inside the op, "RNN Op Changes",
 *            apache/mxnet issue 9543); row b only runs steps t < lengths[b];
 *            the backward direction starts at t = lengths[b]-1.
 *   h0       [L*D, B, Hout] or NULL (zeros);  c0 [L*D, B, H] or NULL (zeros,
 *            LSTM only; must be NULL for GRU).
 *   eps      reserved (no LSTM/GRU cell draws noise); must be NULL.
 *   y        [T, B, D*Hout] output of the last layer; positions t >= lengths[b]
 *            are written as 0.
 *   h_n      [L*D, B, Hout] or NULL; c_n [L*D, B, H] or NULL (LSTM only):
 *            state after each row's last processed step.
 * Returns after enqueueing; a device-side failure (length out of range,
 * barrier timeout) is reported by rnn_get_status.
 */
RCU_API int rnn_forward(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                const float *h0, const float *c0, const float *eps, float *y, float *h_n,
                float *c_n, void *stream);

/*
 * rnn_forward with every buffer in host memory (the same arguments, eps
 * dropped; lengths is a host int32 array).  Nothing is allocated per call
 * beyond staging buffers the handle keeps.
 *   - x and y: when page-locked and registered with CUDA (cudaHostAlloc,
 *     cudaHostRegister, torch pin_memory), the kernels read x and write y in
 *     place through their device addresses over the coherent CPU-GPU link
 *     (NVLink-C2C on Grace-Blackwell): the host<->device transfer happens
 *     inside the packing kernel (x) and the last layer's kernels (y, off the
 *     recurrence's critical path).  Pageable x / y are staged through device
 *     buffers with cudaMemcpyAsync.
 *   - lengths, h0, c0 are copied in, h_n, c_n copied out (small).
 *   - Chunked pipeline (RCU_ATTR_HOST_CHUNKS; automatic from 64 MB of x + y,
 *     one chunk per 64 steps, at most 6): for a unidirectional network
 *     without projection or lengths, with page-locked x and y, the steps
 *     are run in chunks,
 *     each a forward of all layers from every layer's state after the
 *     previous chunk (kept in fp32, so the results equal the unchunked
 *     ones).  x and y then move by cudaMemcpyAsync on two streams the handle
 *     owns, overlapping the other chunks' compute.  rnn_get_pack then
 *     describes the last chunk.
 * Results are in host memory once `stream` has passed this call.  Errors
 * as rnn_forward.
 */
RCU_API int rnn_forward_host(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                             const float *h0, const float *c0, float *y, float *h_n, float *c_n,
                             void *stream);

/*
 * How the last rnn_forward_host call on `h` moved x and y (host pointers to
 * ints, each may be NULL): *chunks = steps chunks of the pipelined form (1 =
 * one forward over all steps); *x_in_place / *y_in_place = 1 when the kernels
 * read x / wrote y through the page-locked host buffer's device address, 0
 * when the data went through device staging buffers and the copy engines.
 * All 0 before the first call.  A description only: no device work.
 */
RCU_API int rnn_host_plan(rcu_rnn_t h, int *chunks, int *x_in_place, int *y_in_place);

/*
 * Backward pass through time (BPTT), the training use of the unrolled cell
 * ("[Feature Request] CUDNN version of RSSM", pytorch/rl issue 366,
 * Motivation; "Integrating CuDNN API for LSTMs with projections",
 * pytorch/pytorch issue 46213, training discussion).  LSTM, GRU and LSTM
 * with projection, uni- or bidirectional, over padded or variable-length
 * batches, with or without cell-state clipping (the clamp passes the
 * gradient where the unclamped cell value lies within the bounds; a
 * projection clip gives RCU_ERR_UNSUPPORTED); on an
 * RCU_BF16 handle, the fp32 gradient of the model with the bf16-rounded
 * weights its forward uses.  Given the forward's inputs x [T,B,in], lengths
 * (device int32 [B], each in [1, T], or NULL = all T; as rnn_forward),
 * h0 [L*D,B,Hout] / c0 [L*D,B,H] (or NULL) and the gradient of a loss with
 * respect to y, dy [T,B,D*Hout] (and to h_n / c_n, dh_n [L*D,B,Hout] / dc_n
 * [L*D,B,H] or NULL = 0), writes the gradients dx [T,B,in], dh0 [L*D,B,Hout]
 * and dc0 [L*D,B,H] (LSTM) — each may be NULL — and keeps the weight
 * gradients of every layer and direction, summed over rows and steps, for
 * rnn_get_weight_grads.  With lengths, row b's steps t >= lengths[b] take no
 * part (as in a packed sequence): dy there is ignored, dx there is 0, h_n /
 * c_n are the states at the row's last step (the reverse direction's at
 * t = 0), and x there is not read.  All device pointers; asynchronous on
 * `stream`; a device-side failure (a wait that ran out, an invalid length)
 * is reported by rnn_get_status.
 * The forward is recomputed inside the call (every layer's output sequence
 * is kept), so only dh_{t-1} = W_hh^T dz_t runs step by step; the rest are
 * GEMMs over all T*B rows.
 */
RCU_API int rnn_backward(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                         const float *h0, const float *c0, const float *dy, const float *dh_n,
                         const float *dc_n, float *dx, float *dh0, float *dc0, void *stream);
/*
 * Weight gradients of layer `layer`, direction `dir` from the last rnn_backward, in the
 * weights' own layout: dW_ih [nG*H, in_l], dW_hh [nG*H, Hout], db_ih, db_hh
 * [nG*H], dW_hr [P, H] (projection only; must be NULL without one).  Any of
 * them may be NULL.  RCU_ERR_STATE before any rnn_backward.
 */
RCU_API int rnn_get_weight_grads(rcu_rnn_t h, int layer, int dir, float *dW_ih, float *dW_hh,
                                 float *db_ih, float *db_hh, float *dW_hr, void *stream);

/*
 * Copy the packing metadata of the last rnn_forward (device int32 buffers):
 *   sorted_idx[B]   original row at sorted position s (length descending,
 *                   equal lengths in ascending row order),
 *   unsorted_idx[B] sorted position of original row b,
 *   batch_sizes[T]  number of rows with length > t.
 * Any pointer may be NULL.
 */
RCU_API int rnn_get_pack(rcu_rnn_t h, int32_t *sorted_idx, int32_t *unsorted_idx, int32_t *batch_sizes,
                 void *stream);

/* Synchronise `stream` and return the device status of the last forward
 * (RCU_OK, RCU_ERR_TIMEOUT or RCU_ERR_LENGTHS), then clear it. */
RCU_API int rnn_get_status(rcu_rnn_t h, void *stream);

/*
 * Clipping of the LSTM state, the cell-state and projection clipping options
 * of cuDNN 7.2 named in "RNN Op Changes" (apache/mxnet issue 9543):
 *   RCU_CLIP_CELL: c_t = clamp(f*c_{t-1} + i*g, lo, hi), before tanh, so the
 *                  clamped value feeds o*tanh(c_t), the next step and c_n;
 *   RCU_CLIP_PROJ: h_t = clamp(W_hr m_t, lo, hi) (LSTMP), the value that feeds
 *                  the next step, y and h_n.
 * enable = 0 turns the target off (lo, hi ignored).  Bounds are used in fp32.
 * Applies to every layer and direction from the next rnn_forward on.
 * Errors: NULL handle, unknown target, lo > hi or NaN -> RCU_ERR_INVALID;
 * GRU handle, or RCU_CLIP_PROJ without projection -> RCU_ERR_UNSUPPORTED.
 */
RCU_API int rnn_set_clip(rcu_rnn_t h, int what, int enable, double lo, double hi);

/* Set a handle attribute (RCU_ATTR_*). */
RCU_API int rnn_set_attr(rcu_rnn_t h, int attr, int64_t value);

/* Number of kernel launches the last rnn_forward enqueued. */
RCU_API int rnn_last_launch_count(rcu_rnn_t h);

/*
 * Per-kernel timing collected while RCU_ATTR_PROFILE is on: entry i (0-based)
 * gives the kernel's name, the summed event-measured duration in ms and the
 * number of launches.  Synchronises on the recorded events.  Returns
 * RCU_ERR_INVALID past the last entry.  rnn_profile_reset clears the totals.
 */
RCU_API int rnn_profile_entry(rcu_rnn_t h, int i, const char **name, double *total_ms,
                              int64_t *count);
RCU_API int rnn_profile_reset(rcu_rnn_t h);

/*
 * Step trace of the first layer's recurrent kernel, recorded while
 * RCU_ATTR_TRACE is on: for each step t < n_steps, 16 global-timer stamps
 * (ns) of CTA 0 are copied to host_out[t*16 .. t*16+15] (0 where a slot is
 * unused).  Tensor-core kernel slots: 0 producer saw the step barrier,
 * 1 first h stage landed, 8 last h stage landed, 2 last MMA issued,
 * 3 epilogue got the accumulator, 5 accumulator read, 11 partner CTA's
 * partial sums received (K split only), 13 gates done, 6 h_t stored,
 * 7 epilogue threads joined, 4 h_t published; slots 9 and 10 hold the MMA
 * thread's clock cycles spent waiting for and issuing h stages.  Portable kernel
 * slots: 0 step start, 1 gates done, 2 barrier passed.  With RCU_ATTR_TRACE
 * = 2 the tensor-core kernel also stamps every CTA for steps 16 .. 23: row
 * T + i*1024 + c holds the stamps of CTA c at step 16 + i (same slots; rows
 * of CTAs past the grid stay 0), so n_steps up to T + 8192 rows are
 * returned.  After an rnn_backward the stamps are instead those of layer 0's
 * reverse-time kernel, row s = reverse step s (time step T-1-s), s <= T.
 * Tensor-core GRU kernel: 0 producer saw every CTA's dR_{t+1}, 1 first dR
 * stage landed, 2 last MMA issued, 3 epilogue got the accumulator,
 * 4 accumulator read and partial sums sent, 5 peers' partial sums received,
 * 6 dR_t published, 7 gradient stores done, 8 next step's activations ready.
 * FFMA kernel: 0 step start, 1 gate gradients done, 2 step barrier passed,
 * 3 W_hh^T dR_t done, 4 partial sums reduced.  Synchronises the stream.
 * host_out is host memory.
 */
RCU_API int rnn_get_trace(rcu_rnn_t h, int64_t *host_out, int n_steps, void *stream);

/* Free the handle, its weights and workspace (synchronises the device). */
RCU_API int rnn_destroy(rcu_rnn_t h);

/* ------------------------------------------------------------------------ */
/* Allocation-free single-layer LSTM                                          */
/* ------------------------------------------------------------------------ */

/* Size of the fixed device scratch behind rnn_lstm_forward_noalloc. */
#define RCU_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * One-layer, one-direction fp32 LSTM forward that allocates no device memory
 * and needs no handle.  It is meant for callers that must not call
 * cudaMalloc themselves or have the library do it: code embedded in a host
 * framework that owns the device heap, processes whose device-memory budget
 * is fixed before they start, and loops that cannot afford an allocation
 * (it may synchronise the device or fail under memory pressure).  The
 * recurrent-cell unroll method this library implements has no counterpart
 * to this entry point: it is an addition for such callers, and computes the
 * same LSTM as rnn_forward with cell RCU_LSTM, one layer, RCU_F32, no lengths.
 *
 *   x [T, B, in_dim]; W_ih [4H, in_dim]; W_hh [4H, H]; b_ih, b_hh [4H] or
 *   NULL (zero); h0, c0 [B, H] or NULL (zero): device, fp32, PyTorch layout.
 *   y [T, B, H]; h_n, c_n [B, H] or NULL: device outputs.
 *
 * Temporary memory comes from a file-scope device array of
 * RCU_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  A problem whose scratch (about 16*T*B*H bytes plus
 * 16*B*H + 16*H) exceeds that size is rejected with RCU_ERR_UNSUPPORTED before
 * any work is enqueued.  All calls share the array and each overwrites it:
 * calls that overlap on the GPU (e.g. on two streams) race.  The first call
 * on a device looks up the array's device address with that device current
 * and caches it.  The call is synchronous (it waits for `stream` and reads
 * the device status back), so it cannot be used while `stream` is being
 * captured into a CUDA graph.  It returns after the work on `stream` has
 * finished: RCU_ERR_TIMEOUT if a device step barrier gave up, RCU_ERR_CUDA for
 * any other launch or device error.
 */
RCU_API int rnn_lstm_forward_noalloc(int T, int B, int in_dim, int hidden, const float *x,
                                     const float *W_ih, const float *W_hh, const float *b_ih,
                                     const float *b_hh, const float *h0, const float *c0,
                                     float *y, float *h_n, float *c_n, void *stream);

/* ------------------------------------------------------------------------ */
/* RSSM prior unroll ("[Feature Request] CUDNN version of RSSM",             */
/* pytorch/rl issue 366, Solution: RSSMPrior and unroll variant 1)           */
/* ------------------------------------------------------------------------ */

/*
 * Create an RSSM prior: state_dim S, action_dim A, hidden Hd (width of the
 * action/state projector and of the prior head's hidden layer), rnn_hidden RH
 * (GRUCell width).  All >= 1 (A >= 0).
 */
RCU_API int rssm_create(rcu_rssm_t *out, int state_dim, int action_dim, int hidden, int rnn_hidden);

/*
 * Copy the prior's weights (device, fp32, PyTorch Linear/GRUCell layout):
 *   W1 [Hd, S+A], b1 [Hd]            action_state_projector (state columns first)
 *   W_ih [3RH, Hd], W_hh [3RH, RH], b_ih, b_hh [3RH]   GRUCell (r, z, n)
 *   W2 [Hd, RH], b2 [Hd]             first Linear of the prior head
 *   W3 [2S, Hd], b3 [2S]             second Linear (first S rows: mean)
 * Biases may be NULL (zero).
 */
RCU_API int rssm_set_weights(rcu_rssm_t h, const float *W1, const float *b1, const float *W_ih,
                     const float *W_hh, const float *b_ih, const float *b_hh, const float *W2,
                     const float *b2, const float *W3, const float *b3, void *stream);

/*
 * RSSM unroll variant 2 ("Given an actor model, we unroll the states for H
 * steps computing the actions on the fly", "[Feature Request] CUDNN version
 * of RSSM", pytorch/rl issue 366, Solution).  The page leaves the actor
 * undefined; it is taken as a deterministic two-layer MLP in the style of the
 * prior's projectors:
 *   action_t = tanh(Wa2 ELU(Wa1 [state_{t-1}, belief_{t-1}] + ba1) + ba2),
 * evaluated on the state and belief before step t (state0/belief0 at t = 0).
 * rssm_set_actor copies the actor (device fp32, row-major): Wa1
 * [actor_hidden, state_dim + rnn_hidden] (state columns first), ba1
 * [actor_hidden], Wa2 [action_dim, actor_hidden], ba2 [action_dim]; NULL bias
 * = zero.  RCU_ERR_UNSUPPORTED if the actor does not fit beside the prior in
 * one cluster's shared memory.
 * rssm_unroll_actor: as rssm_unroll with T = the horizon and no actions
 * input; actions_out [T,B,action_dim] receives the actions (may be NULL).
 * RCU_ERR_STATE before rssm_set_actor.
 */
RCU_API int rssm_set_actor(rcu_rssm_t h, int actor_hidden, const float *Wa1, const float *ba1,
                           const float *Wa2, const float *ba2, void *stream);
RCU_API int rssm_unroll_actor(rcu_rssm_t h, int T, int B, const float *state0,
                              const float *belief0, const float *eps, float *means,
                              float *stds, float *states, float *beliefs, float *actions_out,
                              void *stream);

/*
 * Host-buffer forms of rssm_unroll and rssm_unroll_actor (same arguments, all
 * in host memory).  state0, belief0, actions and eps are copied in; each
 * output that is page-locked and registered with CUDA is written in place by
 * the kernel over the CPU-GPU link, a pageable one is staged and copied back.
 * Results are in host memory once `stream` has passed the call.
 */
RCU_API int rssm_unroll_host(rcu_rssm_t h, int T, int B, const float *state0,
                             const float *belief0, const float *actions, const float *eps,
                             float *means, float *stds, float *states, float *beliefs,
                             void *stream);
RCU_API int rssm_unroll_actor_host(rcu_rssm_t h, int T, int B, const float *state0,
                                   const float *belief0, const float *eps, float *means,
                                   float *stds, float *states, float *beliefs, float *actions_out,
                                   void *stream);

/*
 * Unroll T steps for B independent rows with given actions.  Per step:
 *   a = ELU(W1 [state, action_t] + b1); belief = GRUCell(a, belief);
 *   p = W3 ELU(W2 belief + b2) + b3; mean = p[:S]; std = softplus(p[S:]) + 0.1;
 *   state = mean + eps_t * std.
 *   state0 [B, S], belief0 [B, RH]: device or NULL (zeros).
 *   actions [T, B, A], eps [T, B, S] (the Gaussian noise, supplied by the
 *   caller so the unroll is deterministic): device.
 *   means, stds, states [T, B, S]; beliefs [T, B, RH]: device outputs, the
 *   values after step t's update.
 */
RCU_API int rssm_unroll(rcu_rssm_t h, int T, int B, const float *state0, const float *belief0,
                const float *actions, const float *eps, float *means, float *stds, float *states,
                float *beliefs, void *stream);

/*
 * Backward pass through time of rssm_unroll, the training use of the unroll
 * ("[Feature Request] CUDNN version of RSSM", pytorch/rl issue 366,
 * Motivation).  Takes rssm_unroll's inputs (state0, belief0, actions, eps; as
 * there) and the gradient of a loss with respect to its outputs: dmeans,
 * dstds, dstates [T, B, S] and dbeliefs [T, B, RH], each device or NULL (=
 * 0).  Writes the gradients dstate0 [B, S], dbelief0 [B, RH] and dactions
 * [T, B, A] (each may be NULL) and keeps the weight gradients, summed over
 * rows and steps, for rssm_get_weight_grads.  eps is the noise, an input
 * that is not differentiated.  fp32 throughout; all device pointers;
 * asynchronous on `stream`.  The unroll is recomputed inside the call (a
 * wait that ran out there is reported by rssm_get_status); T, B >= 1.
 */
RCU_API int rssm_backward(rcu_rssm_t h, int T, int B, const float *state0, const float *belief0,
                          const float *actions, const float *eps, const float *dmeans,
                          const float *dstds, const float *dstates, const float *dbeliefs,
                          float *dstate0, float *dbelief0, float *dactions, void *stream);

/*
 * Backward pass through time of rssm_unroll_actor (unroll variant 2: the
 * actions come from the actor set by rssm_set_actor, computed from the
 * state and belief before each step).  As rssm_backward, without actions:
 * dactions [T, B, A] (or NULL) receives the gradient reaching each action
 * the actor produced, the prior's weight gradients are read with
 * rssm_get_weight_grads and the actor's with rssm_get_actor_grads; the
 * actor's input path adds to the gradients of the previous state and
 * belief.  RCU_ERR_STATE without an actor.
 */
RCU_API int rssm_backward_actor(rcu_rssm_t h, int T, int B, const float *state0,
                                const float *belief0, const float *eps, const float *dmeans,
                                const float *dstds, const float *dstates, const float *dbeliefs,
                                float *dstate0, float *dbelief0, float *dactions, void *stream);

/*
 * The actor's weight gradients from the last rssm_backward_actor, in
 * rssm_set_actor's layouts: dWa1 [Ha, S+RH], dba1 [Ha], dWa2 [A, Ha], dba2
 * [A]; device, any may be NULL.  RCU_ERR_STATE when the last backward had no
 * actor.
 */
RCU_API int rssm_get_actor_grads(rcu_rssm_t h, float *dWa1, float *dba1, float *dWa2,
                                 float *dba2, void *stream);

/*
 * Weight gradients of the last rssm_backward in rssm_set_weights' layouts:
 * dW1 [Hd, S+A], db1 [Hd], dW_ih [3RH, Hd], dW_hh [3RH, RH], db_ih, db_hh
 * [3RH], dW2 [Hd, RH], db2 [Hd], dW3 [2S, Hd], db3 [2S]; device, any may be
 * NULL.  RCU_ERR_STATE before any rssm_backward.
 */
RCU_API int rssm_get_weight_grads(rcu_rssm_t h, float *dW1, float *db1, float *dW_ih,
                                  float *dW_hh, float *db_ih, float *db_hh, float *dW2,
                                  float *db2, float *dW3, float *db3, void *stream);

RCU_API int rssm_get_status(rcu_rssm_t h, void *stream);

/* Attributes of an RSSM handle: RCU_ATTR_TRACE (1 = record per-step stamps),
 * RCU_ATTR_BARRIER_TIMEOUT_NS (bound on each wait for a broadcast vector),
 * RCU_ATTR_PROFILE (1 = time named phases), RCU_ATTR_TEST_DROP_ARRIVAL. */
RCU_API int rssm_set_attr(rcu_rssm_t h, int attr, int64_t value);

/*
 * Phase timing collected while RCU_ATTR_PROFILE is on, as rnn_profile_entry:
 * entry i gives the phase's name, its summed event-measured duration in ms
 * and how many times it ran.  Phases: "rssm_unroll" / "rssm_unroll_actor"
 * (the unroll kernel), and in rssm_backward "rssm_bwd_recompute" (everything
 * off the reverse-time chain), "rssm_bwd_chain" (the whole reverse-time
 * sweep, all its launches) and "rssm_bwd_grads" (weight and input gradients).
 * rssm_profile_reset clears the totals.
 */
RCU_API int rssm_profile_entry(rcu_rssm_t h, int i, const char **name, double *total_ms,
                               int64_t *count);
RCU_API int rssm_profile_reset(rcu_rssm_t h);

/*
 * Step trace of the last traced rssm_unroll or rssm_unroll_actor: for each
 * step t < n_steps, 16 stamps of CTA 0 copied to host_out[t*16 ..]: global
 * timer (ns) at slots 0 step start, 5 actor done (rssm_unroll_actor only),
 * 1 phase 1 done, 2 phase 2 done, 3 phase 3 done, 4 phase 4
 * done; SM clock cycles at 8 phase-2 mat-vec done, 9 phase-2 gates done,
 * 10 phase-1 partials done.  Synchronises the stream; host_out is host memory.
 */
RCU_API int rssm_get_trace(rcu_rssm_t h, int64_t *host_out, int n_steps, void *stream);
RCU_API int rssm_last_launch_count(rcu_rssm_t h);
RCU_API int rssm_destroy(rcu_rssm_t h);

#ifdef __cplusplus
}
#endif

#endif /* RCU_H */

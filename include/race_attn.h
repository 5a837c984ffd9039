/*
 * race_attn.h -- C ABI of the GB300 (sm_103a) RACE attention library, librace_attn.so.
 *
 * RACE attention ("RACE Attention" slides, arXiv:2510.04008v5; frames "Soft corner assignments
 * make hashing differentiable", "Each bucket stores mass and a weighted value sum", "Normalize
 * after combining the tables", "Causality is a prefix update of the same statistics"; reading
 * notes sections 2.4-2.6).  For each of L tables with Gaussian hyperplanes W^(l) (P x d):
 *
 *     xhat = x / |x|                                  (each Q and K row; a zero row stays zero)
 *     u^(l)(x) = tanh(W^(l) xhat)                     (P numbers)
 *     phi^(l)_r(x) = softmax_r(beta * u^(l)(x) . v_r) (R = 2^P corners v_r of {-1,+1}^P,
 *                                                      v_{r,t} = +1 iff bit t of r is set)
 *     A^(l) = Phi_K^(l)T V   (R x d, bucket content),   B^(l) = Phi_K^(l)T 1   (R, bucket mass)
 *     O_i = sum_l phi^(l)(Q_i) A^(l) / sum_l phi^(l)(Q_i) B^(l)
 *
 * The causal variant (paper Algorithm 2) replaces A and B by inclusive prefix sums: key t is
 * added to the sketch before query t reads it.
 *
 * Conventions shared by every entry point
 *  - Token tensors Q, K, V, O, dO, dQ, dK, dV are [B, H, N, d], contiguous, d innermost, of
 *    element type `shape->dtype` (float32 or bfloat16), on the current CUDA device, 16-byte
 *    aligned.  Outputs are rounded to nearest-even from float32 arithmetic.
 *  - W is float32 on the device, shared by Q and K and by all tables' rows: one [L, P, d] array
 *    for every (b, h), or, with shape->per_head_w = 1, one set per head, [H, L, P, d], head h
 *    hashing with W[h] for every batch entry (the pages do not say whether heads share their
 *    hyperplanes; both layouts are offered).
 *  - beta is a scalar >= 0: finite, or +INFINITY for hard hashing, the limit the slides name
 *    ("beta -> infinity: hard hashing").  Each bit is then the sign of its projection, and a
 *    row lands in one corner per table.  A projection that is exactly 0 splits the row evenly
 *    over the two corners it separates (the limit sigmoid(0) = 1/2), so a zero row is uniform.
 *    The features are computed as the soft ones at beta = 2^126, which equals the sign rule
 *    exactly for every projection u with |u| >= 2^-119 and at u = 0.  No gradient reaches Q, K,
 *    beta or W (dQ = dK = 0, dbeta = 0, dW = 0); dV is the hard sketch's.  A query whose corners
 *    hold no key in any table has a zero denominator (its output is 0/0), which small inputs can
 *    meet.
 *  - Limits: N >= 1; B * H <= 65535; d a multiple of 8 in [8, 128]; 1 <= P <= 8; 1 <= L <= 16;
 *    L * 2^P <= 256.
 *  - The caller owns every buffer, including `workspace` (size from race_attn_workspace_bytes)
 *    and `state` (size from race_attn_state_bytes).  The library allocates no device memory.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *    stream) and the calls return without synchronising.  Calls that share a workspace must
 *    not overlap on the device.
 *  - Results are deterministic: the same inputs give bitwise identical outputs (fixed-order
 *    reductions, no floating-point atomics).
 *  - Return value: RACE_OK (0) or a negative race_status.  Argument checks happen before any
 *    launch; on an error nothing has been enqueued unless the status is RACE_ERR_CUDA.
 */
#ifndef RACE_ATTN_H
#define RACE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RACE_F32 = 0, RACE_BF16 = 1 } race_dtype;

typedef enum {
    RACE_OK = 0,
    RACE_ERR_INVALID_ARG = -1, /* null pointer, shape or parameter outside the limits above   */
    RACE_ERR_UNSUPPORTED = -2, /* valid arguments this build has no kernel for               */
    RACE_ERR_WORKSPACE = -3,   /* workspace_bytes smaller than race_attn_workspace_bytes()   */
    RACE_ERR_CUDA = -4,        /* a CUDA launch or runtime call failed                        */
    RACE_ERR_ALIGN = -5,       /* a tensor pointer is not 16-byte aligned                     */
    RACE_ERR_SCRATCH_LIMIT = -6, /* race_attn_fwd_noalloc: problem exceeds the built-in scratch */
    RACE_ERR_DEVICE_TIMEOUT = -7, /* race_attn_status: a kernel stopped after a bounded wait    */
    RACE_ERR_NUMERIC = -8,       /* race_attn_status: an output row had a degenerate denominator */
    RACE_ERR_NOALLOC_SETUP = -9  /* the no-alloc scratch could not be set up on this device     */
} race_status;

/* Token-tensor shape and element type, and the layout of W. */
typedef struct {
    int64_t B, H, N, d;
    int32_t dtype;      /* race_dtype */
    int32_t per_head_w; /* 0: W is [L, P, d] for every head; 1: W is [H, L, P, d] */
} race_shape;

/*
 * Bytes of scratch memory race_attn_fwd (is_bwd = 0), race_attn_bwd (is_bwd = 1) or
 * race_attn_bwd with a dW output (is_bwd = 2: also every row's dz / |x|, 8 ((L P + 3) & ~3)
 * bytes per token and (b, h)) needs for this problem.  Returns 0 if the arguments are invalid.  Host function: it launches nothing,
 * but it queries the current device's multiprocessor count (152 when there is no device).
 */
size_t race_attn_workspace_bytes(const race_shape *shape, int L, int P, int causal, int is_bwd);

/*
 * Bytes of the optional saved-sketch buffer `state`: non-causal, the final [A | B] per (b, h)
 * as float32 [B, H, L*2^P, d+1] (columns 0..d-1 = A, column d = B); causal, the sketch at the
 * start of each of the library's sequence segments, float32 [B, H, nseg, L*2^P, d+1], where
 * nseg is a function of the shape and of the current device's multiprocessor count (the work
 * is split to fill the device).  For causal bfloat16 problems with d in {64, 128}, P <= 6,
 * L * P <= 32 and L * 2^P <= 64 the state also holds, after the sketches (each array at the
 * next multiple of 256 bytes), every key's bucket features phi(K_t) as bf16 [B, H, N, F] with
 * F = L * 2^P rounded up to a multiple of 8, and every key's 1 / |K_t| as float32 [B, H, N]:
 * the forward computes them once and the backward reads them instead of recomputing them from
 * K.  Returns 0 if the arguments are invalid.  The same holds for
 * race_attn_workspace_bytes: size buffers with the device current that will run the calls.
 */
size_t race_attn_state_bytes(const race_shape *shape, int L, int P, int causal);

/*
 * Forward pass: O = RACE attention of (Q, K, V) with hyperplanes W and sharpness beta.
 * state: NULL, or a buffer of race_attn_state_bytes() that receives the saved sketch for a
 * later race_attn_bwd call with the same inputs.
 */
int race_attn_fwd(const race_shape *shape, const void *Q, const void *K, const void *V,
                  const float *W, float beta, int L, int P, int causal, void *O, void *state,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass: given the output cotangent dO, writes dQ, dK, dV (all [B, H, N, d]).  The pages
 * print no backward pass; this is the chain rule through the forward's steps ("RACE Attention"
 * slides, frames "Soft corner assignments make hashing differentiable" (Algorithm 1), "Normalize
 * after combining the tables" and, when causal, "Causality is a prefix update of the same
 * statistics" (Algorithm 2)).  With den_i = phi(Q_i) . B and O_i = num_i / den_i:
 *     dnum_i = dO_i / den_i,   dden_i = -(dO_i . O_i) / den_i,
 *     dphi(Q_i) = [A | B] [dnum_i ; dden_i]   (the sketch query i read),
 *     G = sum_i phi(Q_i) [dnum_i | dden_i]   (causal: the suffix sum over i >= j for key j),
 *     dV_j = G_A^T phi(K_j),   dphi(K_j) = G_A V_j + G_B,
 * then, for each Q and K row, the softmax, tanh, projection and normalisation Jacobians.
 * O: the forward output.  It may be NULL: the kernels recompute what they need of O
 * (dO . O per row) from the sketch, which is cheaper than reading it.
 * dbeta: NULL, or device float32 [B, H] (4-byte aligned) that receives d(loss)/d(beta) for each
 * (b, h).  beta is trained with the layer ("RACE Attention" slides, frame "Soft corner
 * assignments make hashing differentiable"); its logits are beta (u . v_r), so every query and
 * key row adds sum_l sum_r ds_r (u . v_r), with ds the softmax gradient of its bucket
 * probabilities.  The gradient of the one shared beta is the sum of the B * H values.  Each
 * value is a sum in a fixed order (per-CTA partials, then a combine), so repeated calls give the
 * same bits.  Overwritten, not accumulated.
 * dW: NULL, or device float32 [B, H, L, P, d] (4-byte aligned) that receives d(loss)/d(W) for
 * each (b, h).  The hyperplanes project the unit rows, z = W x / |x| (slides, frame "Soft corner
 * assignments make hashing differentiable"), so with dz the gradient at z of a Q or K row (the
 * tanh and softmax Jacobians above) d(loss)/d(W) = sum over the Q and K rows of dz (x / |x|)^T.
 * The backward kernels write each row's dz / |x| to the workspace and a reduction forms the sum
 * per (b, h) in a fixed order (repeated calls give the same bits).  A W shared by every head has
 * the sum over b and h as its gradient; a per-head W (per_head_w = 1) the sum over b.  Needs
 * race_attn_workspace_bytes(..., is_bwd = 2) bytes of workspace.  Zero for a hard hash.
 * Overwritten, not accumulated.
 * state: NULL (the sketch is recomputed from K and V), or the buffer a race_attn_fwd call
 * with the same Q, K, V, W, beta, L, P and causal filled in.
 */
int race_attn_bwd(const race_shape *shape, const void *Q, const void *K, const void *V,
                  const float *W, float beta, int L, int P, int causal, const void *O,
                  const void *dO, void *dQ, void *dK, void *dV, float *dbeta, float *dW,
                  const void *state, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Forward pass for callers that cannot allocate device memory (no counterpart in the paper).
 *
 * Some callers are not allowed to call cudaMalloc or to hand the library a workspace: code that
 * runs under an allocator which owns all of the device's memory, or a latency-bound loop that
 * must never allocate because an allocation can synchronise the device.  This entry point
 * computes the same O as race_attn_fwd (same kernels, same arguments, no `state` output) but
 * takes its scratch from a buffer of RACE_NOALLOC_SCRATCH_BYTES (32 MiB) that is compiled into
 * the library as a static device array; every GPU on which the library is loaded holds that
 * buffer until the process exits.  It calls no cudaMalloc, cudaFree or allocating routine.
 *  - Problems whose race_attn_workspace_bytes(shape, L, P, causal, 0) exceeds
 *    RACE_NOALLOC_SCRATCH_BYTES are rejected with RACE_ERR_SCRATCH_LIMIT before any launch.
 *  - Set-up: the driver loads the buffer onto a device when the library first looks up its
 *    address there (under lazy module loading, the CUDA default, not when the library is
 *    loaded).  race_attn_noalloc_init does that for the current device; call it once per device
 *    before a caller's allocator takes the device's memory and before any stream capture.
 *    Otherwise the first race_attn_fwd_noalloc call on the device does it, and returns
 *    RACE_ERR_NOALLOC_SETUP if the device has no room for the buffer or if `stream` is being
 *    captured at that moment.
 *  - All calls on a device share the one buffer and leave their data in it.  Every scratch
 *    element a call reads is written earlier in the same call (its status word is cleared when
 *    it starts), so nothing needs clearing, but two calls that overlap on the GPU (different
 *    streams, or different host threads) race on the buffer and corrupt each other's results:
 *    serialise them.
 *  - Device-side errors (a bounded wait that ran out, a degenerate denominator) are recorded in
 *    the buffer's status word; race_attn_noalloc_status reads it.
 */
#define RACE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int race_attn_fwd_noalloc(const race_shape *shape, const void *Q, const void *K, const void *V,
                          const float *W, float beta, int L, int P, int causal, void *O,
                          void *stream);

/* Sets up the built-in scratch buffer of race_attn_fwd_noalloc on the current device (see
 * there).  Returns RACE_OK (also when it is already set up), RACE_ERR_NOALLOC_SETUP when the
 * device has no room for it, or RACE_ERR_CUDA. */
int race_attn_noalloc_init(void);

/* Device-side status of the last race_attn_fwd_noalloc call on the current device, as
 * race_attn_status reports it for a workspace: synchronises `stream` and reads the status word
 * of the built-in buffer.  RACE_OK when no such call has run on this device. */
int race_attn_noalloc_status(void *stream);

/*
 * One causal decode step per (batch, head): the recurrent form of paper Algorithm 2 ("RACE
 * Attention" slides, frame "Causality is a prefix update of the same statistics").  For every
 * (b, h) the new key k is added to the head's prefix sketch and the new query q reads it:
 *     state[b,h] += phi(k) [v | 1],     o = phi(q) . state[b,h][:, :d] / phi(q) . state[b,h][:, d]
 * shape: N must be 1; q, k, v, o are [B, H, 1, d] of shape->dtype (16-byte aligned).
 * state: float32 [B, H, L * 2^P, d + 1], read and updated in place; race_attn_state_bytes(shape,
 * L, P, 0) bytes.  Zeros start an empty prefix; the `state` that race_attn_fwd with causal = 0
 * fills for a prompt's K and V is the sketch of that prompt, so decoding continues from it.
 * Limits as above (L * P <= 64 follows from them).  No workspace; nothing is allocated.
 */
int race_attn_decode(const race_shape *shape, const void *q, const void *k, const void *v,
                     const float *W, float beta, int L, int P, void *state, void *o, void *stream);

/*
 * Exact angular attention, the kernel RACE attention estimates ("RACE Attention" slides, frame
 * "Choose a nonnegative kernel that can be sketched", paper Eqs. (3)-(4)), in O(N^2):
 *     O_i = sum_j S_ij V_j / sum_j S_ij,   S_ij = (1 - angle(Q_i, K_j) / pi)^gamma
 * over j <= i when causal != 0.  With gamma = P it is the target of the P-bit hash (frame "A
 * hash collision estimates a powered angular kernel"), the reference for measuring the
 * approximation error of race_attn_fwd.  Q, K, V, O as for race_attn_fwd; gamma finite >= 0
 * (0^0 = 1).  A zero row is at angle pi / 2 to every row.  A row whose weights are all zero
 * (every admissible key antipodal) gets 0/0.  Quadratic in N: meant for evaluation sizes.
 * No workspace; nothing is allocated; deterministic.
 */
int race_attn_angular(const race_shape *shape, const void *Q, const void *K, const void *V,
                      float gamma, int causal, void *O, void *stream);

/*
 * Device-side status of the last race_attn_fwd / race_attn_bwd call that used `workspace`.
 * The kernels record two kinds of trouble in the first word of the workspace:
 *  - Kernels that wait for asynchronous (bulk) copies or for each other bound every wait (about
 *    2 s, or 2^22 polls); if a wait runs out they record it and return early, leaving their
 *    outputs incomplete: RACE_ERR_DEVICE_TIMEOUT.
 *  - The forward records an output row whose denominator phi(Q_i) . B is zero, negative or not
 *    finite: the row is then 0/0 or NaN, as the definition gives it (the "Long-context
 *    architectures: Visual walkthrough", Step 6, case A: a query that meets no key mass).  At
 *    float32 this needs every bucket a query can reach to be empty, e.g. beta so large that
 *    sigmoid(-2 beta)^P underflows, or non-finite inputs: RACE_ERR_NUMERIC.
 * This call synchronises `stream`, reads that word and returns RACE_OK, RACE_ERR_DEVICE_TIMEOUT
 * (which takes precedence) or RACE_ERR_NUMERIC (RACE_ERR_CUDA if the stream or the copy
 * failed).  Every fwd/bwd call clears the word when it starts.  race_attn_decode and
 * race_attn_angular take no workspace and report neither.
 */
int race_attn_status(const void *workspace, void *stream);

/*
 * Test hook for the failure path above, not for production use.  While `enable` is non-zero,
 * the causal bfloat16 tcgen05 forward kernel (the one race_attn_fwd and race_attn_fwd_noalloc
 * run for causal bf16 problems with d in {64, 128}, P <= 6, L * P <= 32, L * 2^P <= 64) never
 * requests its first Q / K tiles, so every wait on them runs out: the kernel takes its abort
 * path (drains the copies it did issue, frees its tensor memory) and returns, and the status
 * word reports RACE_ERR_DEVICE_TIMEOUT.  Process-wide; returns RACE_OK.
 */
int race_attn_test_withhold_first_load(int enable);

/* Static description of a status code. */
const char *race_attn_strerror(int status);

/*
 * Instrumentation (host-side, process-wide; off by default).
 * race_attn_launch_count: number of kernels this library has launched so far.
 * race_attn_profile(1) makes every later launch record a CUDA event pair on its stream;
 * race_attn_profile_read(i, ...) synchronises on the recorded events and reports, for kernel
 * name i (0 <= i < count returned), its launches and summed device milliseconds.  Returns the
 * number of distinct kernel names seen, or -1 if i is out of range.  race_attn_profile(0)
 * stops recording; race_attn_profile_reset() clears the table.  Not thread-safe.
 */
uint64_t race_attn_launch_count(void);
int race_attn_profile(int enable);
int race_attn_profile_read(int i, const char **name, int64_t *launches, double *total_ms);
void race_attn_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* RACE_ATTN_H */

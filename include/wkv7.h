/*
 * wkv7.h -- C ABI of the GB300 (sm_103a) WKV7 library, libwkv7.so.
 *
 * The RWKV-7 WKV7 state recurrence, per batch row b and head h, with a state
 * S[N][N] (row i = value index, column j = key index) and, for each token t,
 *
 *     sa_t    = S_{t-1} a_t                                   (pre-update state)
 *     S_t     = S_{t-1} diag(w_t) + sa_t b_t^T + v_t k_t^T
 *     y_t     = S_t r_t                                       (post-update state)
 *
 * Sources (web pages, cited by title and section):
 *   "Foundry/cuda_kernels/timemix.cu" -- file header: WKV7 vectors are
 *     [B][T][H][N] and the state is [B][H][N][N]; k_composites: the two
 *     composite vectors handed to the recurrence are a = -kk, b = kk*a_gate;
 *     tm_fwd_device: one recurrence per (b,h), launched over B*H;
 *     error convention of the extern "C" entries: integer status, no exit.
 *   "infotheory/backends/rwkvzip/rwkv7/model.rs" -- Config::validate: the
 *     head size N is fixed to 64; accumulate_token_step_gradients, WKV kernel
 *     backward: state orientation, y from the post-update state, sa from the
 *     pre-update state, the adjoint implemented by wkv7_backward;
 *     online_train_segment_tbptt: a checkpoint is the state held before a
 *     replay chunk, and the backward replays each chunk forward from it;
 *     module header: single-token streaming inference (wkv7_decode_step).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer to memory the caller allocated and
 *     owns.  The library keeps no pointer after a call returns and allocates
 *     no device memory.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Outputs are valid once the stream reaches
 *     the call.  Gradients are written (=), never accumulated.
 *   - Outputs must not alias inputs or each other (except the in-place state
 *     of wkv7_decode_step).
 *   - r, w, k, v, a, b are fp32 or bf16 (`dtype`); everything else (states,
 *     checkpoints, y, dy and every gradient) is fp32.  Arithmetic is fp32.
 *   - Every pointer must be 16-byte aligned.  Tensors are dense row-major in
 *     the stated layout.
 *   - Return value: WKV7_OK, or a negative code; arguments are checked on
 *     the host before anything is launched, so an error code from argument
 *     checking means nothing ran.  wkv7_last_error() then describes the error
 *     (per calling thread).  WKV7_ECUDA reports a CUDA launch error.
 *   - Results are deterministic: the same inputs give bit-identical outputs
 *     on every run (no atomics, fixed reduction order).
 */
#ifndef WKV7_H
#define WKV7_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { WKV7_F32 = 0, WKV7_BF16 = 1 } wkv7_dtype;

enum {
    WKV7_OK = 0,
    WKV7_EINVAL = -1,       /* bad size, NULL required pointer, misaligned pointer */
    WKV7_ECUDA = -2,        /* a CUDA launch or runtime call failed                 */
    WKV7_EUNSUPPORTED = -3  /* valid request this build cannot serve (e.g. no GPU)  */
};

/* The head size every entry point accepts ("model.rs", Config::validate). */
#define WKV7_HEAD_SIZE 64

/* Number of checkpoints a forward of T tokens writes at stride L: ceil(T/L).
 * Returns -1 if T < 0 or L < 1. */
int wkv7_ckpt_count(int T, int L);

/* Length, in floats, of one (b, h) row of the per-chunk factor cache a
 * forward of T tokens writes: 2048 * ceil(T/16).  Returns -1 if T < 0. */
long long wkv7_factor_floats(int T);

/*
 * Forward over a whole sequence.
 *   B, T, H   batch rows, tokens, heads; B, H >= 1, T >= 0.  N must be 64.
 *   dtype     element type of r, w, k, v, a, b.
 *   r..b      [B][T][H][N] inputs (see the recurrence above).
 *   s0        [B][H][N][N] initial state, or NULL for zeros.
 *   y         [B][T][H][N] output, required when T > 0.
 *   sT        [B][H][N][N] final state, or NULL.
 *   ckpt      [B][H][ceil(T/L)][N][N], or NULL: ckpt[b][h][c] is the state
 *             before token c*L (so ckpt[..][0] = s0).
 *   factors   [B][H][wkv7_factor_floats(T)], or NULL: a cache of per-chunk
 *             quantities of the chunked form (the inverse W, M_k W, Q', W Q_b
 *             and SA of every 16-token chunk) for wkv7_backward to reuse
 *             instead of recomputing them.  Its layout is internal to this
 *             library; only wkv7_backward reads it.  Needs L == 16.
 *   L         checkpoint stride in tokens, L >= 1 (16 is the tuned value).
 * T == 0 writes sT = s0 (or zeros) and nothing else.
 */
int wkv7_forward(int B, int T, int H, int N, wkv7_dtype dtype,
                 const void *r, const void *w, const void *k,
                 const void *v, const void *a, const void *b,
                 const float *s0, float *y, float *sT, float *ckpt,
                 float *factors, int L, void *stream);

/*
 * Backward: the exact adjoint of wkv7_forward, run in reverse time from the
 * checkpoints a forward with the same inputs and the same L wrote.
 *   r..b      the forward's inputs, same dtype and layout.
 *   ckpt      [B][H][ceil(T/L)][N][N] from wkv7_forward (required when T > 0).
 *   factors   the factor cache of that same forward call, or NULL (then the
 *             backward recomputes those quantities).  Needs L == 16.  The
 *             results are the same either way up to fp32 rounding order.
 *   dy        [B][T][H][N] gradient of the loss w.r.t. y (required when T > 0).
 *   dsT       [B][H][N][N] gradient w.r.t. the final state, or NULL for zeros.
 *   dr..db    [B][T][H][N] gradients w.r.t. r, w, k, v, a, b (all required
 *             when T > 0).
 *   ds0       [B][H][N][N] gradient w.r.t. the initial state, or NULL.
 */
int wkv7_backward(int B, int T, int H, int N, wkv7_dtype dtype,
                  const void *r, const void *w, const void *k,
                  const void *v, const void *a, const void *b,
                  const float *ckpt, const float *factors, int L,
                  const float *dy, const float *dsT,
                  float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                  float *ds0, void *stream);

/*
 * One token for each of B*H independent heads (streaming inference).
 *   r..b      [B][H][N] this token's vectors.
 *   state     [B][H][N][N] fp32, read and overwritten in place.
 *   y         [B][H][N] output.
 * Same arithmetic as one step of wkv7_forward.
 */
int wkv7_decode_step(int B, int H, int N, wkv7_dtype dtype,
                     const void *r, const void *w, const void *k,
                     const void *v, const void *a, const void *b,
                     float *state, float *y, void *stream);

/*
 * The producers of w, a and b fused into the recurrence ("Foundry/cuda_kernels/
 * timemix.cu" page: k_decay and k_composites in front of the WKV7 launch,
 * k_wdecay_bwd and k_comp_keymod behind its backward).  Instead of (w, a, b)
 * these entry points take, in the same [B][T][H][N] layout and dtype,
 *   w_pre     the decay pre-activation:  w = exp(-0.606531 * sigmoid(w_pre))
 *   kk        the normalised key:        a = -kk
 *   avec      the in-context gate:       b = kk * avec
 * and compute w, a, b as the inputs are staged, so that they never exist in
 * HBM.  All other arguments are those of wkv7_forward / wkv7_backward.
 * wkv7_forward_fused needs L a multiple of 16 (WKV7_EUNSUPPORTED otherwise).
 * wkv7_backward_fused needs L == 16 and the factor cache of the matching
 * wkv7_forward_fused call (WKV7_EINVAL otherwise, when T > 0), and writes the
 * gradients of the fused inputs in place of (dw, da, db):
 *   dw_pre    dw * w * (-0.606531) * s * (1 - s),  s = sigmoid(w_pre)
 *   dkk       -da + avec * db
 *   davec     kk * db
 * (the terms of k_comp_keymod that pass through a and b; its key-modulation
 * terms belong to the model around the recurrence).  dr, dk, dv and ds0 are
 * as in wkv7_backward.
 */
int wkv7_forward_fused(int B, int T, int H, int N, wkv7_dtype dtype,
                       const void *r, const void *w_pre, const void *k,
                       const void *v, const void *kk, const void *avec,
                       const float *s0, float *y, float *sT, float *ckpt,
                       float *factors, int L, void *stream);
int wkv7_backward_fused(int B, int T, int H, int N, wkv7_dtype dtype,
                        const void *r, const void *w_pre, const void *k,
                        const void *v, const void *kk, const void *avec,
                        const float *ckpt, const float *factors, int L,
                        const float *dy, const float *dsT,
                        float *dr, float *dw_pre, float *dk, float *dv, float *dkk, float *davec,
                        float *ds0, void *stream);

/*
 * The output epilogue of the time-mix block fused into the recurrence
 * ("Foundry/cuda_kernels/timemix.cu" page: k_groupnorm, then k_bonus, after
 * the WKV7 launch; k_bonus_bwd and k_groupnorm_bwd before its backward).  Per
 * token and head, over the head's N outputs y of the recurrence,
 *     o_j = (y_j - mean) / sqrt(var + 64e-5) * gn_w[h][j] + gn_b[h][j]
 *           + (sum_i r_i k_i r_k[h][i]) v_j
 * with mean and the biased variance var of y over the N channels, and the
 * recurrence's own r, k, v.
 *   gn_w, gn_b, r_k  [H][N] fp32: the GroupNorm's per-channel weight and bias
 *                    (one group per head) and the bonus weight.
 *   y                [B][T][H][N] fp32: the recurrence's output, written by the
 *                    forward and read back by the backward.
 *   o                [B][T][H][N] fp32: the epilogue's output.
 * wkv7_forward_gn needs L a multiple of 16 (WKV7_EUNSUPPORTED otherwise);
 * other arguments as in wkv7_forward.  wkv7_backward_gn takes do = dL/do in
 * place of dy, the forward's y, and needs L == 16 and the factor cache of the
 * matching wkv7_forward_gn call (WKV7_EINVAL otherwise, when T > 0).  It
 * writes dr, dw, dk, dv, da, db, ds0 of the whole (recurrence + epilogue;
 * dr, dk, dv include the bonus's own terms) and
 *   dgn_w, dgn_b, dr_k  [H][N] fp32: parameter gradients summed over every
 *                       batch row and token (in a fixed order, no atomics),
 * through a caller-owned workspace of wkv7_gn_workspace_floats(B, H) floats
 * (16-byte aligned; per-(b, h) partial sums).  No fused producers here.
 */
long long wkv7_gn_workspace_floats(int B, int H);
int wkv7_forward_gn(int B, int T, int H, int N, wkv7_dtype dtype,
                    const void *r, const void *w, const void *k,
                    const void *v, const void *a, const void *b,
                    const float *s0, const float *gn_w, const float *gn_b, const float *r_k,
                    float *y, float *o, float *sT, float *ckpt,
                    float *factors, int L, void *stream);
int wkv7_backward_gn(int B, int T, int H, int N, wkv7_dtype dtype,
                     const void *r, const void *w, const void *k,
                     const void *v, const void *a, const void *b,
                     const float *ckpt, const float *factors, int L,
                     const float *y, const float *do_, const float *dsT,
                     const float *gn_w, const float *r_k,
                     float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                     float *ds0, float *dgn_w, float *dgn_b, float *dr_k,
                     float *workspace, void *stream);

/*
 * Sequence parallelism inside one GPU for few, long sequences.  The pages
 * give the recurrence one thread block per (b, h) over all T tokens; these
 * entry points (which have no counterpart there) cut every sequence into
 * nseg equal segments that run side by side, using that the recurrence is
 * affine in the state a segment starts from (S_end = S_start M + Z, M the
 * product of the segment's transitions diag(w_t) + a_t b_t^T):
 *   forward   every segment from I with v = 0 (gives M) and from 0 (gives
 *             Z), a scan S_{k+1} = S_k M_k + Z_k over each head's segments,
 *             then every segment from its start state (y, and checkpoints
 *             and factors kept in the workspace);
 *   backward  every segment's state gradient alone with no gradient at its
 *             end (gives D_k, what it sends to its start), a reverse scan
 *             G_{k-1} = D_k + G_k M_k^T from G = dsT, then every segment with
 *             G_k at its end.
 * The state passes are those of wkv7_forward_state / wkv7_backward_state
 * below.  The split pays off when B*H is small next to the GPU's thread-block
 * slots.
 *   nseg       segments per sequence; T must be a multiple of 16 * nseg.
 *   workspace  device buffer of wkv7_timesplit_workspace_floats(B, T, H,
 *              nseg) floats, 16-byte aligned, owned by the caller; the
 *              backward reads what the matching forward left there, so pass
 *              the same buffer, untouched in between, with the same inputs.
 * Other arguments as in wkv7_forward / wkv7_backward (y required when T > 0,
 * checkpoint stride 16 internally).  Errors as there; WKV7_EINVAL also for a
 * bad nseg, T not a multiple of 16 * nseg, or a missing workspace.
 */
long long wkv7_timesplit_workspace_floats(int B, int T, int H, int nseg);

/*
 * The scan that joins segments, on its own (for segments held elsewhere,
 * e.g. spans of a sequence on other GPUs).  Per (b, h), over k = 0..nseg-1:
 *   backward == 0:  S = init (or 0);  out_k = S;  S = C_k + S M_k;    fin = S
 *   backward != 0:  G = init (or 0);  for k = nseg-1 .. 0: out_k = G;
 *                   G = C_k + G M_k^T;  fin = G
 * M, C, out  [B][nseg][H][N][N] fp32 (M, C, out required);
 * init, fin  [B][H][N][N] fp32, or NULL.  Device pointers, 16-byte aligned.
 */
int wkv7_segment_scan(int B, int H, int nseg, const float *M, const float *C,
                      const float *init, float *out, float *fin, int backward,
                      void *stream);
int wkv7_forward_timesplit(int B, int T, int H, int N, wkv7_dtype dtype,
                           const void *r, const void *w, const void *k,
                           const void *v, const void *a, const void *b,
                           const float *s0, float *y, float *sT,
                           int nseg, float *workspace, void *stream);
int wkv7_backward_timesplit(int B, int T, int H, int N, wkv7_dtype dtype,
                            const void *r, const void *w, const void *k,
                            const void *v, const void *a, const void *b,
                            const float *dy, const float *dsT,
                            float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                            float *ds0, int nseg, float *workspace, void *stream);

/*
 * The state passes alone: the summaries a span of a sequence contributes to
 * the scan above, for spans held in other calls or on other GPUs.  Layouts,
 * ownership, stream order and errors as in wkv7_forward / wkv7_backward.
 *
 * wkv7_forward_state: sT of wkv7_forward for the same w, k, v, a, b and s0,
 * bit-identical (up to the sign of a zero), without y, checkpoints or
 * factors.  v == NULL reads v as zero and k not at all: with s0 = I that is
 * the span's transition product M, with v and s0 = NULL its Z.  sT is
 * required; r is not an input (y is not formed).
 *
 * wkv7_backward_state: ds0 of wkv7_backward for the same r, w, a, b, dy and
 * dsT with the forward's factor cache, bit-identical, without the per-token
 * gradients; with dsT = NULL it is the span's D.  The gradient of the state
 * does not depend on the state itself (nor on k and v), so neither the
 * checkpoints nor k and v are read.
 *   factors  [B][H][wkv7_factor_floats(T)] from wkv7_forward (stride 16) on
 *            the same inputs, required when T > 0;
 *   ds0      [B][H][N][N], required.
 */
int wkv7_forward_state(int B, int T, int H, int N, wkv7_dtype dtype,
                       const void *w, const void *k, const void *v,
                       const void *a, const void *b,
                       const float *s0, float *sT, void *stream);
int wkv7_backward_state(int B, int T, int H, int N, wkv7_dtype dtype,
                        const void *r, const void *w, const void *a, const void *b,
                        const float *factors, const float *dy, const float *dsT,
                        float *ds0, void *stream);

/* Largest B*H*ceil(T/16) that wkv7_forward_backward_noalloc accepts. */
#define WKV7_NOALLOC_MAX_CHUNK_HEADS 4096

/*
 * Forward followed by backward in one call that allocates no memory at all.
 * This entry point is a library convenience; the method's description has
 * no counterpart to it.
 *
 * It is for callers that cannot call cudaMalloc or hand out temporary device
 * buffers: code that runs under a host framework with a fixed, pre-planned
 * memory pool, inside a real-time loop where allocation is forbidden, or from
 * a language binding with no CUDA allocator of its own.  wkv7_forward +
 * wkv7_backward with a factor cache need a caller-owned workspace (the cache,
 * wkv7_factor_floats(T) floats per (b, h)); here that workspace is a
 * fixed-size array inside the library instead.
 *
 * The call runs exactly the tuned path: wkv7_forward with checkpoint stride
 * 16 writing the factor cache into the library's array, then wkv7_backward
 * reading it.  The caller passes every input and output:
 *   r..b, s0, dy, dsT, y, sT, dr..db, ds0   as in wkv7_forward / wkv7_backward
 *   ckpt      [B][H][ceil(T/16)][N][N] checkpoints (stride 16), required when
 *             T > 0; written by the forward half, read by the backward half.
 * Limits and sharing:
 *   - B*H*ceil(T/16) must not exceed WKV7_NOALLOC_MAX_CHUNK_HEADS (the array
 *     is 4096 * 8 KiB = 32 MiB); larger requests return WKV7_EINVAL with a
 *     message naming the limit.
 *   - Every GPU that loads this library holds that 32 MiB until the process
 *     exits.
 *   - All calls on a device share the one array.  Each call writes every
 *     entry it later reads, so nothing needs clearing, but two calls whose
 *     work overlaps on the GPU (different streams, no ordering between them)
 *     race on it and give wrong results.
 *   - The first call on a device looks up the array's device address once
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 */
int wkv7_forward_backward_noalloc(int B, int T, int H, int N, wkv7_dtype dtype,
                                  const void *r, const void *w, const void *k,
                                  const void *v, const void *a, const void *b,
                                  const float *s0, const float *dy, const float *dsT,
                                  float *y, float *sT, float *ckpt,
                                  float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                                  float *ds0, void *stream);

/*
 * One training step in one call: wkv7_forward (checkpoint stride 16, with
 * the factor cache when `factors` is given) followed by wkv7_backward on the
 * same batch.  This entry point is a library convenience; the method's
 * description has no counterpart to it.  Every head is independent in both
 * directions, so the batch is cut into `nsplit` contiguous blocks of batch
 * rows; each block runs its forward and then its backward on a stream of
 * its own: block 0 on `stream` itself, the others on streams of the library,
 * forked from `stream` by an event and joined back into it.  A block's backward starts as soon as its forward is done, while the
 * other blocks' forwards finish, which keeps more of the GPU busy than the
 * two calls in a row.  Results are bit-identical to those two calls.
 *   r..b, s0, dy, dsT, y, sT, dr..db, ds0   as in wkv7_forward / wkv7_backward
 *   ckpt      [B][H][ceil(T/16)][N][N], required when T > 0: written by the
 *             forward half, read by the backward half.
 *   factors   [B][H][wkv7_factor_floats(T)] or NULL (the backward half then
 *             rebuilds the per-chunk factors itself).
 *   nsplit    number of blocks, 0 (the library's default: 4 when B*H is at
 *             least 512, else 2) to 4; more blocks than batch rows means one
 *             row per block, 1 runs the two calls in order on `stream` itself.
 * Ownership and errors as in wkv7_forward: the caller owns every buffer;
 * every argument is checked (WKV7_EINVAL, WKV7_EUNSUPPORTED) before anything
 * is launched; WKV7_ECUDA on a launch or stream error, after which the
 * library's streams are still joined back into `stream`.  The library
 * creates its streams and events when a call first needs them (at most three
 * streams and four events per device) and keeps them for the life of the
 * process; concurrent calls from several host threads are serialised while
 * they enqueue their work.
 *
 * wkv7_forward_backward_blocks: the number of blocks a call of any of the
 * three one-call forms makes for these B, T, H and nsplit (each block
 * launches one forward and one backward; the _gn form adds one reduction),
 * or -1 for B or H < 1, T < 0 or nsplit outside 0 .. 4.  Host only.
 */
int wkv7_forward_backward_blocks(int B, int T, int H, int nsplit);
int wkv7_forward_backward(int B, int T, int H, int N, wkv7_dtype dtype,
                          const void *r, const void *w, const void *k,
                          const void *v, const void *a, const void *b,
                          const float *s0, const float *dy, const float *dsT,
                          float *y, float *sT, float *ckpt, float *factors,
                          float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                          float *ds0, int nsplit, void *stream);

/*
 * The same one-call training step through wkv7_forward_fused and
 * wkv7_backward_fused: (w_pre, kk, avec) in place of (w, a, b) and
 * (dw_pre, dkk, davec) in place of (dw, da, db), as described there.  The
 * factor cache is required when T > 0 (WKV7_EINVAL otherwise), since the
 * fused backward reads it.  Everything else is as in wkv7_forward_backward,
 * results bit-identical to the two fused calls.
 */
int wkv7_forward_backward_fused(int B, int T, int H, int N, wkv7_dtype dtype,
                                const void *r, const void *w_pre, const void *k,
                                const void *v, const void *kk, const void *avec,
                                const float *s0, const float *dy, const float *dsT,
                                float *y, float *sT, float *ckpt, float *factors,
                                float *dr, float *dw_pre, float *dk, float *dv, float *dkk, float *davec,
                                float *ds0, int nsplit, void *stream);

/*
 * The same one-call training step through wkv7_forward_gn and
 * wkv7_backward_gn (the GroupNorm + bonus output epilogue): do = dL/do in
 * place of dy, the epilogue's weights gn_w, gn_b, r_k ([H][N]), its output o,
 * its parameter gradients dgn_w, dgn_b, dr_k ([H][N], summed over every batch
 * row and token) and the workspace of wkv7_gn_workspace_floats(B, H) floats,
 * as described there; the factor cache is required when T > 0.  Each block
 * leaves the per-(b, h) parameter-gradient sums of its rows in the workspace,
 * and one reduction over all B rows follows on `stream` once the blocks are
 * joined, in the same order as wkv7_backward_gn's: results bit-identical to
 * the two calls.  Everything else as in wkv7_forward_backward.
 */
int wkv7_forward_backward_gn(int B, int T, int H, int N, wkv7_dtype dtype,
                             const void *r, const void *w, const void *k,
                             const void *v, const void *a, const void *b,
                             const float *s0, const float *do_, const float *dsT,
                             const float *gn_w, const float *gn_b, const float *r_k,
                             float *y, float *o, float *sT, float *ckpt, float *factors,
                             float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                             float *ds0, float *dgn_w, float *dgn_b, float *dr_k,
                             float *workspace, int nsplit, void *stream);

/*
 * Status of the kernels' asynchronous copies on the current device.  The
 * kernels stage their inputs with bulk copies whose completion they wait for
 * a bounded time; a wait that runs out (which no correct run should see) sets
 * a per-device flag instead of hanging the GPU.  This call waits for the
 * device to finish its work, returns WKV7_ECUDA (and clears the flag) if any
 * launch since the last check set it, WKV7_OK otherwise.  The library looks
 * up the flag's device address on its first forward, backward or status call
 * on each device.
 */
int wkv7_async_status(void);

/* Text of the last error on the calling thread ("" if none). */
const char *wkv7_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_H */

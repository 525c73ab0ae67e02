/*
 * retention.h -- C ABI of libretention.so: RetNet multi-scale retention on
 * one NVIDIA B300 (sm_103a).
 *
 * The operation (per batch row b and head h, 0-based positions n, m):
 *
 *   out[b,h,n,:] = sum_{m <= n} gamma_h^(n-m) * (q[b,h,n,:] . k[b,h,m,:]) / sqrt(dk) * v[b,h,m,:]
 *
 * i.e. O = ((Q K^T / sqrt(dk)) (.) D_h) V with the causal decay matrix
 * D_h[n,m] = gamma_h^(n-m) for n >= m and 0 otherwise, and the recurrent state
 *
 *   S[b,h] = sum_m gamma_h^(N-1-m) k[b,h,m,:]^T v[b,h,m,:]      (dk x dv)
 *
 * Sources: "RetNet Guide: Retentive Networks & The Impossible Triangle",
 * sections "3. Multi-Scale Retention (MSR)" (gamma_h = 1 - 2^(-5-h)),
 * "1. The Parallel Representation ..." (D and R = ((QK^T) (.) D) V),
 * "2. The Recurrent Representation ..." (S_n = gamma S_{n-1} + K_n^T V_n,
 * R_n = Q_n S_n), "3. The Chunkwise Recurrent Representation ..." (chunk
 * state carry and the zeta_j = gamma^(j+1) cross-chunk weight) and
 * "1. PyTorch Implementation of MultiScaleRetention" (0-based heads, the
 * 1/sqrt(d) scaling of the query).  The factor 1/sqrt(dk) multiplies the
 * query only; states hold unscaled k^T v sums, so a state produced by
 * retention_chunkwise can be advanced by retention_step.
 *
 * Beyond the forward: retention_backward gives the gradients of the forward
 * (the pages print none; they are the derivatives of the definition above),
 * retention_rotate the position phase rotation of queries and keys
 * ("2. Relative Position via Complex Exponential Phase Rotations"), and
 * retention_groupnorm / retention_chunkwise_groupnorm the per-head GroupNorm
 * of the multi-scale retention output ("1. The Parallel Representation ...").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All data pointers are DEVICE pointers on the current CUDA device, owned by
 *   the caller, 16-byte aligned, dense and row-major:
 *     q, k  [B][H][N][dk]       v, out  [B][H][N][dv]      (sequence calls)
 *     q, k  [B][H][dk]          v, out  [B][H][dv]         (step calls)
 *     state, state_out  [B][H][dk][dv]  float32
 *     gamma  [H]  float32, each value in [0, 1]
 * - Element type: the base names take bfloat16 q, k, v, out (and dout and
 *   the gradients); the *_f32 names take float32.  Accumulation is float32
 *   everywhere.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *   asynchronous: they enqueue work on `stream` and never synchronise the
 *   device.  Inputs must stay valid until that work has run.
 * - out must not alias q, k or v.
 * - Return value: RET_OK, or a negative ret_status.  Argument checks run on
 *   the host before anything is enqueued; on a non-OK return nothing was
 *   enqueued (except RET_ERR_CUDA, where a launch may have been attempted).
 * - A device-side wait in the tensor-core kernels that exceeds its time
 *   limit sets a bit in the library's device status word (see
 *   retention_device_status) and the kernel returns; outputs are then
 *   undefined.
 */
#ifndef RETENTION_H
#define RETENTION_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RET_OK = 0,
    RET_ERR_INVALID = -1,     /* null pointer, size < 0 (or 0 where not allowed), misaligned pointer */
    RET_ERR_UNSUPPORTED = -2, /* valid arguments outside what the kernels handle (shape, chunk) */
    RET_ERR_CUDA = -3         /* a CUDA runtime call or a kernel launch failed */
} ret_status;

/* Device status bits (retention_device_status). */
#define RET_DEV_WAIT_TIMEOUT 0x1u /* a bounded barrier wait gave up */

/*
 * retention_chunkwise -- chunkwise recurrent forward, bf16 q/k/v/out.
 *
 * Per "3. The Chunkwise Recurrent Representation ...": the sequence is cut
 * into chunks of `chunk` tokens; inside a chunk the parallel form runs on the
 * tensor cores, and a float32 state S (dk x dv) is carried from chunk to
 * chunk as S <- gamma^L S + sum_j gamma^(L-1-j) k_j^T v_j (L = chunk length;
 * the last chunk may be shorter when N % chunk != 0).  The state starts at
 * zero.  If state_out is not NULL it receives the state after token N-1
 * (zero when N == 0).
 *
 * Supported: chunk in {32, 64, 128}; dk a multiple of 16 in [16, 512]; dv a
 * multiple of 16 in [16, 1024]; N >= 0.  Other shapes return
 * RET_ERR_UNSUPPORTED.  The chunk length is a tiling choice that does not
 * change the result (every chunk length computes the same sums, up to
 * rounding order), so the kernels pick their tile height, 64 or 128 tokens,
 * from the sizes whatever chunk is asked for: 128 (the tensor cores' full
 * tile height), unless 64-token tiles give more CTAs (a short sequence with
 * few heads); above 256 query/key columns the tiles are 512 columns wide,
 * 64 tokens high, with 64-wide value tiles.  Widths below the kernel's tile
 * (128, 256 or 512 query and key columns, 64 or 128 value columns) are
 * padded with zeros by the loads, which leaves every product unchanged.  The work is cut into units,
 * one per (batch row, head, value tile).  With fewer units than SMs every
 * unit's sequence is split into segments; with more, only the units of the
 * last, partial wave are split (so that wave holds about one CTA per SM).
 * When the call splits sequences it allocates a float32 scratch buffer for
 * the segment states stream-ordered (cudaMallocAsync / cudaFreeAsync on
 * `stream`); retention_chunkwise_ws takes a caller-provided buffer instead.
 */
int retention_chunkwise(const void *q, const void *k, const void *v, const float *gamma,
                        void *out, float *state_out,
                        int B, int H, int N, int dk, int dv, int chunk, void *stream);

/*
 * retention_chunkwise_from_state -- retention_chunkwise continued from a
 * given state: the recurrence of "3. The Chunkwise Recurrent Representation
 * ..." started from S_{-1} = state_in instead of zero, so that a sequence
 * processed in pieces (chunked prefill) gives the same outputs and final
 * state as one call on the whole sequence:
 *
 *   out_t  = scale [ sum_{m<=t} gamma^(t-m) (q_t . k_m) v_m + gamma^(t+1) q_t state_in ]
 *   S_N-1  = gamma^N state_in + sum_m gamma^(N-1-m) k_m^T v_m         (scale = 1/sqrt(dk))
 *
 * state_in: float32 [B][H][dk][dv] row-major in device memory (the layout of
 * state_out, e.g. the state_out of a call on the preceding tokens), 16-byte
 * aligned, read only, owned by the caller; NULL means zero (then this is
 * retention_chunkwise).  It must not overlap state_out (the call reads it
 * while the last segment of the sequence writes state_out): state_in ==
 * state_out returns RET_ERR_INVALID.  When N == 0, state_out receives a copy
 * of state_in.  Everything else (shapes, workspace, errors) is as for
 * retention_chunkwise.
 */
int retention_chunkwise_from_state(const void *q, const void *k, const void *v, const float *gamma,
                                   const float *state_in, void *out, float *state_out,
                                   int B, int H, int N, int dk, int dv, int chunk, void *stream);

/*
 * retention_chunkwise_rotated -- retention_chunkwise_from_state of the queries
 * and keys turned by the position phase rotation of "2. Relative Position via
 * Complex Exponential Phase Rotations" (as retention_rotate below, with the
 * same theta and n0 for q and k).  With one value tile per head (dv of at
 * most 64, or exactly 128), the rotation is fused into the kernels' load
 * stage: each Q/K tile is turned in shared memory after it lands and before
 * the tensor cores read it, so q and k are read from HBM once and the turned
 * copies are never written.  With several value tiles per head (each would
 * turn the same Q/K tiles) that fusion measured slower than separate
 * passes, so q and k are turned into a
 * stream-ordered scratch buffer (cudaMallocAsync / cudaFreeAsync on
 * `stream`) by the standalone rotation first.  Either way:
 *
 *   out = chunkwise(rotate(q, theta, n0), rotate(k, theta, n0), v, gamma; state_in)
 *
 * The turned pairs are rounded to bf16 (as retention_rotate's output would
 * be).  theta: float32 [dk/2] device memory, 4-byte aligned; n0 >= 0 the
 * position of token 0; state_in nullable as for
 * retention_chunkwise_from_state (it must not equal state_out).  Shapes and
 * the workspace as for retention_chunkwise; n0 plus N rounded up to the tile
 * length (64, or 128 for chunk 128) must not exceed 2^24 (positions exact in
 * float32), else RET_ERR_UNSUPPORTED.
 */
int retention_chunkwise_rotated(const void *q, const void *k, const void *v, const float *gamma,
                                const float *theta, int n0, const float *state_in, void *out,
                                float *state_out, int B, int H, int N, int dk, int dv, int chunk,
                                void *stream);

/*
 * retention_rotate -- the position phase rotation of queries or keys: "2.
 * Relative Position via Complex Exponential Phase Rotations" multiplies the
 * query and key of token n by e^(i n theta), so that their product depends on
 * n - m only.  Pairs (2j, 2j+1) of the d real dimensions are one complex
 * coordinate with frequency theta_j; with the real dot product that the
 * retention calls use, queries and keys are both turned by a = (n0 + n) theta_j:
 *
 *   y[2j] = x[2j] cos a - x[2j+1] sin a,   y[2j+1] = x[2j] sin a + x[2j+1] cos a
 *
 * so rotate q and k with the same theta and n0 before retention_chunkwise,
 * retention_parallel or retention_step (n0 = the position of the sequence's
 * first token, e.g. the number of tokens already in the state).  x, y: bf16
 * [B][H][N][d], 16-byte aligned device memory; y may be x (in place), other
 * overlaps are not allowed.  theta: float32 [d/2] device memory (learnable on
 * the pages; any values).  d must be a multiple of 8, n0 >= 0 and
 * n0 + N <= 2^24 (else RET_ERR_UNSUPPORTED).  Angles are reduced modulo 2 pi in
 * fp32 before the sine and cosine.  Asynchronous on `stream`.
 */
int retention_rotate(const void *x, const float *theta, void *y,
                     int B, int H, int N, int d, int n0, void *stream);

/*
 * retention_groupnorm -- the normalisation of the heads' outputs that
 * multi-scale retention applies before its output projection: "1. The
 * Parallel Representation for High-Throughput Pretraining", MSR(X) =
 * GroupNorm(Concat(R_1, ..., R_H)) W_O, with one group per head over the
 * concatenated channels ("1. PyTorch Implementation of MultiScaleRetention").
 * For every batch row b, token n and head h, over the dv channels c:
 *
 *   mu = mean_c r[b][h][n][c],   var = mean_c (r[b][h][n][c] - mu)^2
 *   y[b][n][h][c] = (r[b][h][n][c] - mu) / sqrt(var + eps) * weight[h dv + c] + bias[h dv + c]
 *
 * r: bf16 [B][H][N][dv] (the retention output layout); y: bf16 [B][N][H][dv]
 * (heads concatenated per token); both 16-byte aligned device memory and must
 * not overlap.  weight, bias: float32 [H dv] device memory, or NULL for one and
 * zero.  eps >= 0 (the pages use 1e-6).  Statistics in fp32.  dv must be a
 * multiple of 4, at most 1024, and B H at most 65535 (else
 * RET_ERR_UNSUPPORTED).  Asynchronous on `stream`; N == 0 is a no-op.
 */
int retention_groupnorm(const void *r, const float *weight, const float *bias, void *y,
                        int B, int H, int N, int dv, float eps, void *stream);

/*
 * retention_chunkwise_groupnorm -- retention_chunkwise with the normalisation
 * of multi-scale retention fused into its output epilogue: "1. The Parallel
 * Representation for High-Throughput Pretraining", MSR(X) =
 * GroupNorm(Concat(R_1, ..., R_H)) W_O, one group per head ("1. PyTorch
 * Implementation of MultiScaleRetention").  `out` receives, with the heads
 * concatenated per token ([B][N][H][dv] bf16, the layout of
 * retention_groupnorm's y),
 *
 *   out[b][n][h][c] = (R[c] - mu) / sqrt(var + eps) * weight[h dv + c] + bias[h dv + c]
 *
 * where R is the fp32 retention output row of (b, h, n) (before any bf16
 * rounding) and mu, var its mean and biased variance over the dv channels.
 * weight, bias: float32 [H dv], 16-byte aligned device memory, or NULL (one,
 * zero).  eps >= 0.  state_out as for retention_chunkwise (the plain state).
 * Supported when dv is 64 or 128 (a head's row is then one value tile of one
 * CTA), with the chunk sizes and dk of retention_chunkwise; otherwise
 * RET_ERR_UNSUPPORTED (use retention_chunkwise then retention_groupnorm).
 * Workspace as for retention_chunkwise.
 */
int retention_chunkwise_groupnorm(const void *q, const void *k, const void *v, const float *gamma,
                                  const float *weight, const float *bias, float eps,
                                  void *out, float *state_out,
                                  int B, int H, int N, int dk, int dv, int chunk, void *stream);

/*
 * retention_chunkwise_workspace_size -- bytes of scratch retention_chunkwise_ws
 * needs for this shape (0 when the plan does not split the sequence).
 * Host only; returns RET_ERR_INVALID / RET_ERR_UNSUPPORTED like
 * retention_chunkwise would.
 */
int retention_chunkwise_workspace_size(int B, int H, int N, int dk, int dv, int chunk,
                                       size_t *bytes);

/*
 * retention_chunkwise_ws -- retention_chunkwise with caller-owned scratch:
 * `workspace` is a device buffer of `workspace_bytes` bytes, 256-byte
 * aligned, used only by the work this call enqueues.  No memory is allocated.
 * retention_chunkwise_workspace_size gives the size of the preferred plan.
 * With less, a call whose last partial wave would be split runs those units
 * whole instead (same results; that wave takes longer); a call that needs
 * the scratch for every unit (fewer units than SMs) and gets less returns
 * RET_ERR_INVALID.  `workspace` may be NULL with workspace_bytes 0.
 */
int retention_chunkwise_ws(const void *q, const void *k, const void *v, const float *gamma,
                           void *out, float *state_out,
                           int B, int H, int N, int dk, int dv, int chunk,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * retention_chunkwise_noalloc -- retention_chunkwise for callers that must not
 * allocate device memory.  The paper has no counterpart to this entry point;
 * it exists for callers such as serving runtimes that plan all device memory
 * at start-up under a fixed budget (an allocation on the request path can
 * fail, stall or fragment the pool) and embedders whose host code may not call
 * the CUDA allocator.  Same arguments, layout and results as
 * retention_chunkwise; it allocates and frees nothing.
 *
 * Scratch: the segment states live in a file-scope device array of
 * 8 MiB (8388608 bytes) that every GPU loading the library reserves until the
 * process exits.  The call runs the plan retention_chunkwise_ws runs with
 * 8 MiB of workspace: where retention_chunkwise would cut the units of a last,
 * partial wave (see retention_chunkwise_ws) and their states need more, those
 * units run whole instead.  Shapes whose plan needs more scratch than that
 * even so (fewer units than SMs, every unit cut) return RET_ERR_UNSUPPORTED
 * before anything is enqueued.  Nothing in the array has to start at zero: each call
 * writes every slot it later reads, so stale contents of an earlier call are
 * never used.
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) once; make that first call
 * before any stream capture.  A lookup that fails returns RET_ERR_CUDA and is
 * tried again by the next call on that device; a successful one is kept.
 * Concurrency: every call on a device shares the one array, so calls whose
 * work overlaps on the GPU (different streams, or different host threads
 * without ordering) race on it; order them on one stream or serialise them.
 */
int retention_chunkwise_noalloc(const void *q, const void *k, const void *v, const float *gamma,
                                void *out, float *state_out,
                                int B, int H, int N, int dk, int dv, int chunk, void *stream);

/*
 * retention_chunkwise_host -- retention_chunkwise with q, k, v, out and
 * state_out in HOST memory (same shapes and layouts; gamma, H float32, is a
 * device pointer).  The (batch row, head) pairs are cut into up to 8 slabs
 * (whole batch rows; with B == 1, equal groups of heads); each slab is copied
 * to the device, run by the chunkwise kernels and copied back on one of
 * three streams the library creates per device on the first call (make it
 * outside stream capture), so the copies in the two directions and the
 * kernels of successive slabs overlap.  The streams are forked from and
 * joined back to `stream` with events: the call is ordered on `stream` and
 * only enqueues work, so the host buffers must stay valid, and out/state_out
 * unread, until `stream` has reached that point.  Page-locked host memory
 * (cudaHostAlloc / cudaHostRegister) is needed for the copies to overlap;
 * pageable memory gives the same results, serialised.  state_out may be NULL.
 * dev_buffer: NULL (a device buffer is allocated stream-ordered on `stream`)
 * or a 256-byte aligned device buffer of dev_buffer_bytes >= the size from
 * retention_chunkwise_host_buffer_size.  Supported shapes: those of
 * retention_chunkwise.  Each slab is planned on its own (its own split into
 * segments), so results can differ from retention_chunkwise's in rounding
 * order, within the same error bound.
 */
int retention_chunkwise_host(const void *q_host, const void *k_host, const void *v_host, const float *gamma,
                             void *out_host, float *state_out_host,
                             int B, int H, int N, int dk, int dv, int chunk,
                             void *dev_buffer, size_t dev_buffer_bytes, void *stream);
/* Device bytes retention_chunkwise_host needs for these sizes (three slab
 * slots: q, k, v, out, state and segment scratch of one slab each).  Host only. */
int retention_chunkwise_host_buffer_size(int B, int H, int N, int dk, int dv, int chunk, size_t *bytes);

/*
 * retention_chunkwise_launches -- number of kernels one retention_chunkwise
 * call with these sizes enqueues (for launch accounting).  Host only.
 */
int retention_chunkwise_launches(int B, int H, int N, int dk, int dv, int chunk, int *launches);

/*
 * retention_chunkwise_f32 -- the chunkwise form with float32 q/k/v/out on the
 * CUDA cores (plain fp32 FMA, no TF32).  chunk in [1, 128]; dk, dv in
 * [1, 256]; the per-block working set must fit in shared memory, else
 * RET_ERR_UNSUPPORTED.
 */
int retention_chunkwise_f32(const float *q, const float *k, const float *v, const float *gamma,
                            float *out, float *state_out,
                            int B, int H, int N, int dk, int dv, int chunk, void *stream);

/*
 * retention_parallel / retention_parallel_f32 -- the parallel form
 * ("1. The Parallel Representation ..."): O = ((QK^T/sqrt(dk)) (.) D) V over
 * the whole sequence, no state; O(N^2) work, the training form of the pages.
 * retention_parallel with dk a multiple of 16 in [16, 256] and dv a multiple
 * of 16 in [16, 1024] runs on the tensor cores: per 128-row query tile a
 * causal loop over 128-row key tiles, S = Q K_j^T and O += P~ V_j as
 * tcgen05 MMAs (bf16 operands, fp32 accumulation in tensor memory), the decay
 * gamma^(n-m) and 1/sqrt(dk) applied to S in registers; a key tile is skipped
 * only where its largest decay factor is exactly zero in fp32.  Other widths
 * (dk, dv in [1, 256]) and the float32 twin run tiled on the CUDA cores.
 * N >= 0.
 */
int retention_parallel(const void *q, const void *k, const void *v, const float *gamma,
                       void *out, int B, int H, int N, int dk, int dv, void *stream);
int retention_parallel_f32(const float *q, const float *k, const float *v, const float *gamma,
                           float *out, int B, int H, int N, int dk, int dv, void *stream);

/*
 * retention_step / retention_step_f32 -- one recurrent decode step for every
 * (b, h) ("2. The Recurrent Representation ..."):
 *   S[b,h] <- gamma_h S[b,h] + k[b,h]^T v[b,h]     (in place, float32)
 *   out[b,h] = (q[b,h] / sqrt(dk)) S[b,h]          (the updated state)
 * There is no gamma argument: gamma_h = 1 - 2^(-5-h) for the 0-based head
 * index h, rounded once to float32 (the values retention_gamma_schedule
 * returns).  dv must be a multiple of 4; dk >= 1.
 */
int retention_step(const void *q, const void *k, const void *v, float *state, void *out,
                   int B, int H, int dk, int dv, void *stream);
int retention_step_f32(const float *q, const float *k, const float *v, float *state, float *out,
                       int B, int H, int dk, int dv, void *stream);

/*
 * retention_step_rotated -- retention_step for the token at position `pos`,
 * with q and k turned by the position phase rotation (theta float32 [dk/2],
 * as retention_rotate) as they are loaded, in float32, before the state
 * update: the decode step that continues a sequence prefilled by
 * retention_chunkwise_rotated (pos = the number of tokens before it, n0
 * included).  0 <= pos < 2^24 and dk even, else RET_ERR_UNSUPPORTED.
 */
int retention_step_rotated(const void *q, const void *k, const void *v, const float *theta, int pos,
                           float *state, void *out, int B, int H, int dk, int dv, void *stream);

/*
 * retention_backward -- gradients of the forward (any of its forms: they
 * compute one function), for training.  "3. The Chunkwise Recurrent
 * Representation ..." gives the chunkwise form as the way to train on long
 * sequences but prints no gradient; these are the partial derivatives of the
 * forward started from state_in (S0),
 *
 *   out_n = s [ sum_{m<=n} g^(n-m) (q_n . k_m) v_m + g^(n+1) q_n S0 ],
 *   S_N   = g^N S0 + sum_m g^(N-1-m) k_m^T v_m          (s = 1/sqrt(dk), g = gamma[h]),
 *
 * for the loss <dout, out> + <dstate, S_N>:
 *
 *   dq_n  = s [ sum_{m<=n} g^(n-m) (dout_n . v_m) k_m + g^(n+1) S0 dout_n ]
 *   dk_m  = s sum_{n>=m} g^(n-m) (dout_n . v_m) q_n + g^(N-1-m) dstate v_m
 *   dv_m  = s sum_{n>=m} g^(n-m) (q_n . k_m) dout_n + g^(N-1-m) k_m dstate
 *   dS0   = s sum_n g^(n+1) q_n^T dout_n + g^N dstate
 *
 * q, k, dq, dk: bf16 [B][H][N][dk]; v, dout, dv: bf16 [B][H][N][dv]; gamma:
 * float32 [H]; state_in, dstate, dstate_in: float32 [B][H][dk][dv]; all
 * row-major device memory, 16-byte aligned, owned by the caller.  state_in
 * and dstate may be NULL (zero); dstate_in may be NULL (not written).  The
 * gradients are written, not accumulated.  Outputs must not overlap inputs or
 * one another: a gradient whose bytes overlap q, k, v, dout or another
 * gradient, or dstate_in equal to dstate or state_in, returns
 * RET_ERR_INVALID.  When N == 0, dstate_in receives a copy of dstate (zero if
 * NULL).
 * How it runs: with bf16 tensors and dk, dv multiples of 16 in [16, 512], on
 * the tensor cores, each gradient as a chunkwise forward of permuted
 * operands (dq the forward of (dout, v, k) from S0^T; dk and dv the
 * time-reversed forwards of (v, dout, q) and (k, q, dout) from dstate^T/(s g)
 * and dstate/(s g); dS0 = s g times the final state of the latter), with bf16
 * operands and float32 accumulation and state.  The forwards read q, k, v
 * and dout in place and write the gradients in place (the time-reversed ones
 * take the rows from the last to the first); a stream-ordered scratch buffer
 * (cudaMallocAsync / cudaFreeAsync on `stream`) holds the starting states
 * and segment states.  The three forwards run concurrently on `stream` and
 * two streams the library creates per device on its first gradient call
 * (forked from and joined back to `stream` with events, so the call is
 * ordered on `stream` like any other and can be captured in a CUDA graph;
 * make the first call on a device outside stream capture).  Otherwise (other widths, or the float32 twin) float32 arithmetic
 * on the CUDA cores, one launch, no workspace.  Supported: dk, dv multiples of
 * 4, at most 512; other widths return RET_ERR_UNSUPPORTED.
 * retention_backward_f32 is the same with float32 q/k/v/dout/dq/dk/dv.
 */
int retention_backward(const void *q, const void *k, const void *v, const float *gamma,
                       const float *state_in, const void *dout, const float *dstate,
                       void *dq, void *dk_out, void *dv_out, float *dstate_in,
                       int B, int H, int N, int dk, int dv, void *stream);
int retention_backward_f32(const float *q, const float *k, const float *v, const float *gamma,
                           const float *state_in, const float *dout, const float *dstate,
                           float *dq, float *dk_out, float *dv_out, float *dstate_in,
                           int B, int H, int N, int dk, int dv, void *stream);

/*
 * retention_backward_launches -- number of kernels one bf16 retention_backward
 * call with these sizes enqueues (for launch accounting); the flags say
 * whether state_in and dstate are given and dstate_in is wanted.  Host only.
 */
int retention_backward_launches(int B, int H, int N, int dk, int dv, int has_state_in, int has_dstate,
                                int want_dstate_in, int *launches);

/*
 * retention_gamma_schedule -- host function: gamma_out[h] = 1 - 2^(-5-h),
 * h = 0..H-1, rounded to float32 ("3. Multi-Scale Retention (MSR)",
 * 0-based heads).  gamma_out is HOST memory of H floats.
 */
int retention_gamma_schedule(int H, float *gamma_out);

/*
 * retention_device_status -- copies the library's device status word of the
 * current device into *flags (RET_DEV_* bits; 0 = no fault seen) and clears
 * it when `clear` is non-zero.  Synchronises the device.
 */
int retention_device_status(unsigned int *flags, int clear);

/*
 * retention_test_stall_waits -- host function for tests of the failure path
 * (no counterpart on the pages).  With `microseconds` > 0, every later
 * launch of the tensor-core chunkwise kernel (retention_chunkwise and the
 * calls built on it) makes one barrier wait that nothing completes, with
 * that limit; the wait gives up, sets RET_DEV_WAIT_TIMEOUT in the device
 * status word, and every role of the CTA unwinds exactly as after a real
 * timeout (loads and MMAs in flight are waited for, tensor memory is
 * released) and the kernel returns.  Outputs of such calls are undefined.
 * 0 turns it off (the default).  The setting is process-wide and is read
 * when a call enqueues its kernels.  microseconds above 10 000 000 return
 * RET_ERR_INVALID.
 */
int retention_test_stall_waits(unsigned int microseconds);

/* retention_status_string -- static text for a ret_status value. */
const char *retention_status_string(int status);

/* retention_version -- ABI version (major * 100 + minor). */
int retention_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RETENTION_H */

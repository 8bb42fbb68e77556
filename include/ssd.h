/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 chunked SSD forward library.
 *
 * The operation is the chunked state-space-duality (SSD) forward pass of
 * "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)"
 * (dbyun.net/article/14364).  For every batch row b and head h, with
 * g = h / (nheads / ngroups) the head's B/C group:
 *
 *     h_t = exp(A[h] dt_t) h_{t-1} + dt_t x_t B_t^T        (state, headdim x dstate)
 *     y_t = h_t C_t + D[h] x_t                              (section "Mamba-2 架构")
 *
 * computed chunk by chunk (chunk_size T tokens) in three stages: the
 * within-chunk log2 cumsum G (section "Kernel 1"), the chunk-to-chunk state
 * pass (section "Kernel 2: fwd_pass_state") and the fused chunk output
 * (section "Kernel 3: compute_out").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers: all tensor pointers are DEVICE pointers owned by the caller.
 *   The library never allocates, frees or retains them beyond the call.
 *   Every tensor is contiguous, row-major, 16-byte aligned.
 * Layouts (B = batch, L = seqlen, H = nheads, P = headdim, S = dstate,
 *   G = ngroups, nc = ceil(L / T)):
 *     x, y            [B, L, H, P]   dtype of the call (bf16 or f32)
 *     Bm, Cm          [B, L, G, S]   dtype of the call
 *     dt              [B, L, H]      f32, already activated (softplus etc. is
 *                                    the caller's job)
 *     A, D            [H]            f32 (A < 0 for a decaying state)
 *     G_cum, dt_t     [B, H, L]      f32, token-contiguous (the layout the
 *                                    pages move decay_cumsum and dt to)
 *     init_state, final_state  [B, H, P, S]      f32
 *     chunk_states    [B, H, nc, P, S]          f32; chunk_states[:,:,c] is
 *                                    the state before token c*T, so
 *                                    chunk_states[:,:,0] == init_state
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Every call is asynchronous and stream-ordered.
 * Errors: every call validates its arguments on the host BEFORE launching
 *   anything and returns a status; nothing aborts, throws or prints.  A
 *   failed launch returns SSD_ERR_CUDA.  Errors raised inside a kernel (a
 *   bounded wait that ran out) are recorded in a per-device status word that
 *   ssd_stream_status() reads.
 * Threads: calls are thread-safe; the only shared host state is a
 *   mutex-guarded cache of TMA descriptors and tuning choices.
 * Device lifetime: the library caches, per device, the device addresses of
 *   its own __device__ arrays (the status word, the scratch array of
 *   ssd_fwd_noalloc) for the life of the process; do not use it on a device
 *   after cudaDeviceReset has been called there.
 * Supported sizes: 1 <= P <= 256, 1 <= S <= 512, 1 <= T <= 256, H % G == 0,
 *   L >= 0 (L == 0 copies init_state to final_state and launches nothing
 *   else).  The tensor-core (tcgen05) kernels serve bf16 with T a multiple
 *   of 128: the state pass for P in {64, 128} and S % 64 == 0; the chunk
 *   output for P == 64 and S in {64, 128, 256}, and for S in {384, 512}
 *   with T == 128; the one-head fused pass for P == 64 and S in
 *   {64, 128, 256, 384, 512} (at 384 / 512 B and C stream through it in
 *   128-row dstate blocks); the head-pair fused pass for P == 64, S in
 *   {64, 128} and an even number of heads per group.  ssd_fwd takes a fused
 *   pass wherever one serves the shape, except at S 384 / 512 when every
 *   chunk state is asked for (the staged path writes them as part of its
 *   work, and is faster there).  Other shapes and all f32 calls run
 *   f32-arithmetic CUDA-core kernels.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,  /* null pointer, bad size or inconsistent dims */
    SSD_ERR_UNSUPPORTED = 2,  /* sizes outside the supported ranges above */
    SSD_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
    SSD_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    SSD_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
    SSD_ERR_WORKSPACE = 6     /* workspace pointer missing or too small */
} ssd_status_t;

typedef enum {
    SSD_BF16 = 0,  /* x, Bm, Cm, y are bf16; arithmetic accumulates in f32 */
    SSD_F32 = 1    /* x, Bm, Cm, y are f32; all arithmetic is f32 */
} ssd_dtype_t;

typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
} ssd_dims_t;

/*
 * Stage 1 -- within-chunk cumulative decay (section "Kernel 1").
 *   G_cum[b,h,t] = log2(e) * sum_{t' = c*T}^{t} A[h] * dt[b,t',h],  c = t / T.
 * The sum restarts at every chunk boundary.  G is kept in log2 units so the
 * later stages use exp2.  dt_t (may be NULL) receives dt transposed to
 * [B, H, L].
 */
ssd_status_t ssd_chunk_cumsum(const float *dt, const float *A, float *G_cum, float *dt_t,
                              ssd_dims_t dims, int chunk_size, void *stream);

/*
 * Stage 2 -- chunk-to-chunk state pass (section "Kernel 2: fwd_pass_state").
 * For c = 0 .. nc-1, per (b, h):
 *     chunk_states[b,h,c] = h
 *     h <- exp2(G_last) h + X_c^T (B_c * dt_c * exp2(G_last - G_c))      ([P,S])
 * where G_last is G at the chunk's last VALID token (a ragged last chunk
 * uses its own last token, not a zero-padded one).  h starts at init_state
 * (NULL = zeros).  final_state (may be NULL) receives h after the last chunk.
 * chunk_states may be NULL when only the final state is wanted.
 */
ssd_status_t ssd_state_pass(const void *x, const void *Bm, const float *dt_t, const float *G_cum,
                            const float *init_state, float *chunk_states, float *final_state,
                            ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, void *stream);

/*
 * Stage 3 -- chunk output (section "Kernel 3: compute_out").  Per (b, c, h):
 *     Y = exp2(G) * (C_c h_c^T) + (exp2(G_i - G_j) * (C_c B_c^T) * M) (dt * X_c) + D[h] X_c
 * with M the inclusive causal mask (i >= j) and h_c = chunk_states[b,h,c].
 * The T x T score matrix never leaves the chip.  Masked entries are zero,
 * never inf or NaN.
 */
ssd_status_t ssd_chunk_out(const void *x, const void *Bm, const void *Cm, const float *dt_t,
                           const float *G_cum, const float *chunk_states, const float *D, void *y,
                           ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, void *stream);

/*
 * Stages 2 and 3 fused (bf16 tensor-core path): walks every (batch, head)
 * sequence once, carrying the state on chip from tile to tile, and writes y,
 * the final state (may be NULL) and, if chunk_states is not NULL, every
 * chunk's start state.  Arithmetic is that of ssd_state_pass followed by
 * ssd_chunk_out.  G_cum and dt_t are stage 1's outputs.  Long sequences are
 * cut into segments processed in parallel; each segment starts from the
 * state its predecessor leaves in `workspace` (at least
 * ssd_state_out_workspace_size bytes, 256-byte aligned; contents on entry do
 * not matter).  Returns SSD_ERR_UNSUPPORTED for f32 calls and for shapes
 * outside the tensor-core path (see "Supported sizes"); use the two separate
 * stages there.
 */
ssd_status_t ssd_state_out(const void *x, const void *Bm, const void *Cm, const float *dt_t,
                           const float *G_cum, const float *D, const float *init_state, void *y,
                           float *final_state, float *chunk_states, ssd_dims_t dims,
                           ssd_dtype_t dtype, int chunk_size, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Workspace bytes ssd_state_out needs (depends on the current device's SM count). */
size_t ssd_state_out_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size);

/* Which kernels ssd_fwd runs for these arguments (chunk_size 0 = auto). */
typedef enum {
    SSD_PATH_INVALID = -1,
    SSD_PATH_STAGED_CUDA_CORES = 0,   /* cumsum -> state_pass -> chunk_out, f32 CUDA cores */
    SSD_PATH_STAGED_TENSOR_CORES = 1, /* cumsum -> state_pass -> chunk_out, tcgen05 */
    SSD_PATH_FUSED_TENSOR_CORES = 2,  /* cumsum -> state_out (fused), tcgen05 */
    SSD_PATH_FUSED_PAIR_TENSOR_CORES = 3 /* one fused kernel, two heads of a group per CTA,
                                            G formed in the kernel; tcgen05 */
} ssd_path_t;
ssd_path_t ssd_fwd_path(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, int want_chunk_states);

/*
 * Bytes of device workspace ssd_fwd needs for these arguments (the G_cum,
 * dt_t and, when the caller does not want them, the chunk states the
 * three-stage path keeps between stages, plus the chain buffers of the fused
 * path).  chunk_size 0 means "let the library choose", as in ssd_fwd: once
 * the choice for the shape is fixed (ssd_fwd_chosen_chunk_size), that
 * choice's size; before, without chunk states, the largest size among the
 * candidates the tuner may time (candidates on CUDA cores are left out where
 * another candidate runs on tensor cores: the tuner skips a candidate whose
 * workspace does not fit).  Returns 0 for invalid arguments.
 */
size_t ssd_fwd_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                              int want_chunk_states);

/*
 * Whole forward pass: stage 1 -> 2 -> 3 on one stream, or the fused
 * single-pass kernel (state carried on chip / in L2 between chunks) when the
 * shape allows it.  y receives the output; final_state and chunk_states are
 * optional outputs (NULL = not wanted); init_state may be NULL (zeros).
 * chunk_size 0 lets the library choose among {64, 128, 256} (see
 * ssd_fwd_chosen_chunk_size: the first such call for a shape may time the
 * candidates on the caller's buffers and stream).
 * workspace must hold ssd_fwd_workspace_size(dims, dtype, chunk_size,
 * chunk_states != NULL) bytes, 256-byte aligned; its contents on entry do
 * not matter.  On the head-pair path (SSD_PATH_FUSED_PAIR_TENSOR_CORES) with
 * few head pairs, that size covers the prefilled-segment plan, which also
 * holds G and dt_t; a workspace too small for it that still holds the plan
 * whose segments hand their states to one another is accepted, and that
 * plan runs (SSD_ERR_WORKSPACE below both).
 */
ssd_status_t ssd_fwd(const void *x, const float *dt, const float *A, const void *Bm,
                     const void *Cm, const float *D, const float *init_state, void *y,
                     float *final_state, float *chunk_states, ssd_dims_t dims,
                     ssd_dtype_t dtype, int chunk_size, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * Backward pass: gradients of the forward (ssd_fwd's y and final state) with
 * respect to every input, for a scalar loss whose gradients with respect to
 * y and the final state are dy [B, L, H, P] (call dtype) and dfinal
 * [B, H, P, S] f32 (NULL = zero).  The pages name the backward pass but do
 * not give it; it is the adjoint of the recurrence of section "Mamba-2 架构"
 * worked chunk by chunk (64-token chunks) like the forward:
 *   a reverse state pass carries the state gradient from the last chunk to
 *   the first, dh_in = exp(L_T) dh_out + sum_i exp(L_i) dy_i C_i^T, and each
 *   (batch, chunk, head) then forms its dx, ddt, dB, dC, dA, dD terms from
 *   the chunk's start state (recomputed by the forward state pass) and the
 *   gradient of its end state.
 * Outputs (caller-owned device memory, every one written):
 *   dx [B, L, H, P] (call dtype), ddt [B, L, H] f32, dA [H] f32, dB, dC
 *   [B, L, G, S] (call dtype; summed over the heads of each group), dD [H]
 *   f32, dinit [B, H, P, S] f32 (may be NULL: not wanted; the gradient with
 *   respect to init_state, or to the zero initial state when init_state is
 *   NULL).
 * Arithmetic: bf16 calls with P == 64 and S in {64, 128} run tcgen05 kernels
 * (128-token chunks, bf16 operands, f32 accumulation); every other call runs
 * f32 arithmetic on CUDA cores (bf16 inputs widened).  Supported: P <= 64
 * and the sizes of ssd_fwd; other headdims return SSD_ERR_UNSUPPORTED.
 * workspace: ssd_bwd_workspace_size(dims, dtype) bytes, 256-byte aligned;
 * contents on entry do not matter.
 */
size_t ssd_bwd_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype);
ssd_status_t ssd_bwd(const void *x, const float *dt, const float *A, const void *Bm,
                     const void *Cm, const float *D, const float *init_state, const void *dy,
                     const float *dfinal, void *dx, float *ddt, float *dA, void *dB, void *dC,
                     float *dD, float *dinit, ssd_dims_t dims, ssd_dtype_t dtype,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gated RMS norm, the gating and normalisation that follow the scan (the
 * post's operator-fusion section names gating, normalisation and the output
 * projection after the scan; gate and norm run here as one pass, the
 * projection is a plain GEMM).  Per token, over each group of group_size
 * consecutive channels of the token's dim = nheads * headdim channels:
 *     g   = y * silu(z),  silu(z) = z / (1 + exp(-z))
 *     out = g / sqrt(mean(g^2 over the group) + eps) * weight
 * y, z, out: [ntokens, dim] in the call's dtype (e.g. ssd_fwd's y viewed as
 * [B*L, H*P]); weight: [dim] f32.  out may be y or z (in place).  Arithmetic
 * f32.  Only element alignment is required; 16-byte aligned buffers with
 * group_size a multiple of 8 (bf16) or 4 (f32) take 16-byte vectors.
 * dim % group_size != 0 or eps < 0 returns SSD_ERR_INVALID_ARG.
 */
ssd_status_t ssd_gated_rmsnorm(const void *y, const void *z, const float *weight, void *out,
                               int64_t ntokens, int64_t dim, int64_t group_size, float eps,
                               ssd_dtype_t dtype, void *stream);

/*
 * Single-token decode step on a carried state (section "Mamba-2 架构": the
 * recurrence for one token, i.e. how a final state from ssd_fwd is used
 * during generation).  dims.seqlen must be 1; per (b, h), g = h / (H / G):
 *     state[p,s] <- exp(A[h] dt[b,h]) state[p,s] + dt[b,h] x[b,h,p] Bm[b,g,s]
 *     y[b,h,p]    = sum_s Cm[b,g,s] state[p,s] + D[h] x[b,h,p]
 * (the state after the update feeds y, as in the chunked forward).
 * Layouts are those of the forward with L = 1: x, y [B, 1, H, P], dt [B, 1, H],
 * Bm, Cm [B, 1, G, S], state_in / state_out [B, H, P, S] f32.  state_out may
 * be state_in (in-place update) or a separate buffer; partly overlapping
 * buffers return SSD_ERR_INVALID_ARG.  Unlike the other entry points this
 * one asks only for element alignment (a token's slice of a [B, L, ...]
 * tensor is rarely 16-byte aligned); 16-byte aligned state and B / C with
 * dstate % 4 == 0 take the vectorised kernel.  Arithmetic is f32 (inputs
 * widened, exp of the decay in f32); y is rounded to the call's dtype.
 */
ssd_status_t ssd_decode_step(const void *x, const float *dt, const float *A, const void *Bm,
                             const void *Cm, const float *D, const float *state_in,
                             float *state_out, void *y, ssd_dims_t dims, ssd_dtype_t dtype,
                             void *stream);

/*
 * ssd_fwd without a workspace argument, for callers that cannot allocate
 * device memory (code running inside an allocator or memory-pool callback, a
 * host framework that owns all device allocations, a latency-critical loop
 * that must not pay for an allocation's implicit synchronisation).  The
 * pages describe no counterpart; this is a convenience of this library.
 *
 * The workspace is a fixed scratch array inside the library: 160 MiB
 * (167772160 bytes) per device, reserved on a device when the library's code
 * for this entry point is first loaded there and kept until the process
 * exits.  A call whose least workspace exceeds it returns
 * SSD_ERR_UNSUPPORTED before launching anything: ssd_fwd_workspace_size(...),
 * or on the head-pair path the smaller of its two plans' scratch (see
 * ssd_fwd).  Roughly: the one-head fused path needs 8 bytes per batch x
 * head x token; the staged paths also hold the chunk states when
 * chunk_states is NULL.  Inputs, outputs and their
 * conventions are exactly those of ssd_fwd, and nothing is allocated.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before capturing
 * a stream into a CUDA graph.  Every call on a device shares the same array
 * and it keeps the previous call's contents (no region needs to start at
 * zero), so calls whose kernels may overlap on the GPU -- concurrent streams,
 * or several host threads -- race on it: serialize them.
 */
ssd_status_t ssd_fwd_noalloc(const void *x, const float *dt, const float *A, const void *Bm,
                             const void *Cm, const float *D, const float *init_state, void *y,
                             float *final_state, float *chunk_states, ssd_dims_t dims,
                             ssd_dtype_t dtype, int chunk_size, void *stream);

/*
 * ssd_fwd from host memory to host memory.  x, dt, A, Bm, Cm, D, init_state
 * (optional) and the outputs y and final_state (optional) are HOST buffers
 * in ssd_fwd's layouts; page-locked (pinned) host memory lets the copies run
 * asynchronously.  workspace is DEVICE memory of at least
 * ssd_fwd_host_workspace_size(dims, dtype, chunk_size) bytes, 256-byte
 * aligned.  Chunk states are not returned (use ssd_fwd for those).
 *
 * The sequence is cut into up to four parts of whole chunks (at least 512
 * tokens each); part k runs ssd_fwd on its tokens from the state part k-1
 * ended with -- "Kernel 2: fwd_pass_state" carries the state across chunk
 * boundaries, so this computes ssd_fwd's function, up to the rounding of the
 * carried state.  Part k's inputs are copied up on one internal stream while
 * part k-1 computes on `stream` and part k-2's y is copied down on a second
 * internal stream, so both copy directions overlap the kernels.  The call is
 * asynchronous and stream-ordered: it starts after the work already on
 * `stream`, and `stream` waits for all of it -- also when an error is
 * returned after some copies started -- so the host buffers must stay
 * untouched until `stream` has completed (synchronize it before reading y).  The internal streams and events of each device are created
 * on first use and kept; calls are serialized by a mutex while they issue
 * work (not while it runs).  Errors: as ssd_fwd, plus SSD_ERR_WORKSPACE for
 * a short or unaligned workspace and SSD_ERR_CUDA for a failed copy.
 */
size_t ssd_fwd_host_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size);
ssd_status_t ssd_fwd_host(const void *x, const float *dt, const float *A, const void *Bm,
                          const void *Cm, const float *D, const float *init_state, void *y,
                          float *final_state, ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Chunk size ssd_fwd uses for chunk_size == 0 with these dims and dtype
 * (0 for invalid arguments).  The pages search the best configuration per
 * shape ("Accelerating Mamba-2 forward-pass kernels with CUDA Tile
 * (cuTile)", section "Mamba-2 性能优化"); here the choice among {64, 128, 256}
 * -- and, on the head-pair path, between its prefilled-segment and hand-off
 * plans -- is fixed once per (batch, seqlen, nheads, headdim, dstate,
 * ngroups, dtype) and process, by whichever comes first:
 *   - the first ssd_fwd(chunk_size = 0) call without chunk_states, outside
 *     stream capture, whose y and final_state overlap no input: it runs
 *     every candidate whose workspace fits the one passed, once untimed and
 *     twice between CUDA events on the caller's stream, synchronizing that
 *     stream (so that first call blocks the host and takes a few times a
 *     forward), keeps the fastest, then runs the call itself;
 *   - this function, or any other ssd_fwd(chunk_size = 0) call: the static
 *     choice (128 for bf16; for f32 64 when seqlen <= 64, else 128).
 * A fixed choice never changes in the process, so chunk_states can be sized
 * from this function.  Make the first chunk_size = 0 call for a shape
 * before any stream capture that could be active in another thread (the
 * tuner records and waits on events).
 */
int ssd_fwd_chosen_chunk_size(ssd_dims_t dims, ssd_dtype_t dtype);

/* 1 if the choice above was fixed by timing the candidates, else 0. */
int ssd_fwd_chunk_size_was_timed(ssd_dims_t dims, ssd_dtype_t dtype);

/*
 * Sequence-sharded (context-parallel) forward, one segment of the sequence
 * per rank, ranks in sequence order.  Section "Kernel 2: fwd_pass_state"
 * makes the state at the end of one call the initial state of the next, and
 * the state update is linear in the state, so the segments need one
 * exchange of a per-segment summary:
 *   1. ssd_segment_summary on every rank: seg_state [B, H, P, S] f32 = the
 *      segment's end state when run from a zero state, and seg_decay [B, H]
 *      f32 = the segment's total decay sum_t A[h] dt[b,t,h] in log2 units
 *      (log2(e) times the natural-log sum; the pages keep G in log2 units).
 *      Inputs as for ssd_fwd (x, dt, A, Bm of the segment).  workspace:
 *      ssd_segment_summary_workspace_size(dims, dtype, chunk_size) bytes,
 *      256-byte aligned (G and dt^T of the segment).
 *   2. the caller all-gathers (seg_state, seg_decay) of every segment.
 *   3. ssd_carry_in on rank r: h_in = exp2(D_{r-1}) h_{r-1} + s_{r-1} with
 *      h_0 = init_state (NULL: zeros); seg_states [n_segments, B, H, P, S]
 *      and seg_decays [n_segments, B, H] hold the gathered summaries (only
 *      the first `upto` segments are read; upto = r).  h_in [B, H, P, S]
 *      f32 may be init_state itself, but may not overlap anything else.
 *      Only batch, nheads, headdim and dstate of dims are used.
 *   4. ssd_fwd of the segment with init_state = h_in: y, final state and
 *      chunk states of that segment (chunk states match the unsharded run's
 *      when every segment but the last is a whole number of chunks).
 * Errors as ssd_fwd; every call is asynchronous on `stream`.
 */
size_t ssd_segment_summary_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size);
ssd_status_t ssd_segment_summary(const void *x, const float *dt, const float *A, const void *Bm,
                                 float *seg_state, float *seg_decay, ssd_dims_t dims,
                                 ssd_dtype_t dtype, int chunk_size, void *workspace,
                                 size_t workspace_bytes, void *stream);
ssd_status_t ssd_carry_in(const float *seg_states, const float *seg_decays,
                          const float *init_state, int n_segments, int upto, float *h_in,
                          ssd_dims_t dims, void *stream);

/*
 * Number of kernel launches this library has issued in this process (all
 * devices, all threads).  Diagnostic: a call rejected by validation leaves it
 * unchanged; the benchmark reports launches per step from it.
 */
uint64_t ssd_launch_count(void);

/* Static, human-readable name of a status. */
const char *ssd_status_string(ssd_status_t status);

/*
 * Synchronizes `stream`, then reads and clears the calling thread's current
 * device's kernel status word.  Returns SSD_ERR_TIMEOUT if any kernel since
 * the last read gave up a bounded wait, SSD_ERR_CUDA if the stream reports
 * an error, else SSD_OK.
 * Fault injection (debug only): with SSD_FAULT_SKIP_ARRIVE=1 in the
 * environment when the head-pair kernel is launched, one compute warp per
 * CTA skips a barrier arrival on the CTA's first tile and every wait of that
 * launch gives up after 20 ms; the launch then records the timeout here,
 * leaves with nothing in flight, and its outputs are undefined.
 */
ssd_status_t ssd_stream_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */

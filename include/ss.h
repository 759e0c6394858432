/*
 * ss.h -- C ABI of the GB300 (sm_103a) Mamba-1 selective scan.
 *
 * The operation (baracuda-kernels `selective_scan.rs`, module doc
 * "Algorithm summary"), per batch b, channel d and state n:
 *
 *   delta_eff = softplus(delta[b,t,d] + delta_bias[d])     (bias and softplus optional)
 *   dA        = exp(delta_eff * A[d,n])
 *   h[n]      = dA * h[n] + delta_eff * B[b,t,n] * u[b,t,d]  (h starts at zero)
 *   y[b,t,d]  = (sum_n h[n] * C[b,t,n] + D[d] * u[b,t,d]) * silu(z[b,t,d])  (D, z optional)
 *   last_state[b,d,n] = h[n] after t = L-1
 *
 * softplus(x) = log(1 + e^x), silu(z) = z / (1 + e^-z).
 *
 * Layouts ("Shape contract" of the same page): every tensor is contiguous and
 * row-major.  u, delta, z, y, dy: [Bsz, L, Dch].  A: [Dch, N].  B, C:
 * [Bsz, L, N].  D, delta_bias: [Dch].  last_state: [Bsz, Dch, N].
 *
 * Element types.  "io" tensors (u, delta, B, C, z, y, dy) are f32, f16 or
 * bf16 as selected by `dtype`.  A, D, delta_bias, last_state and every gradient are
 * f32.  Arithmetic and the recurrence state are f32.
 *
 * Ownership and execution.  Every pointer is caller-owned DEVICE memory of
 * the current CUDA device.  The library allocates nothing, never
 * synchronises and enqueues all work on `stream` (a cudaStream_t passed as
 * void*; NULL is the legacy default stream).  Returning SS_OK means the work
 * was enqueued; a fault during execution surfaces at the caller's next
 * synchronisation.  Inputs are read only; outputs are fully overwritten (no
 * caller zeroing is needed); input and output ranges must not overlap.
 * Calls may come from several host threads and devices at once: a call's
 * state lives in its arguments and workspace, except the library-owned
 * scratch of ss_fwd_noalloc (see there).
 *
 * Errors are reported before anything is launched; nothing is written then.
 * Results are deterministic: the same arguments on the same GPU give
 * bit-identical outputs, forward and backward (no atomics anywhere).
 */
#ifndef SS_H
#define SS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element-type ids of the io tensors; the numbering follows the dtype ids of
 * the `..._workspace_bytes(.., dtype_id)` query on the baracuda-kernels page
 * (0 = f32, 1 = f16, 2 = bf16). */
typedef enum { SS_F32 = 0, SS_F16 = 1, SS_BF16 = 2 } ss_dtype;

/* Status codes; the first three mirror the page's error kinds
 * (Unsupported, InvalidProblem, WorkspaceTooSmall). */
typedef enum {
    SS_OK = 0,
    SS_ERR_INVALID_PROBLEM = 1,     /* negative extent, missing required pointer, optional-term mismatch */
    SS_ERR_UNSUPPORTED = 2,         /* dtype, N outside {1,2,4,8,16,32}, size limit, pointer not 16-byte aligned */
    SS_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the matching *_workspace_bytes() query */
    SS_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
    SS_ERR_DEVICE_TIMEOUT = 5,      /* from ss_device_status: a kernel gave up waiting for its tile copies */
    SS_ERR_STAGING_FALLBACK = 6     /* from ss_device_status: a kernel could not use TMA (results intact) */
} ss_status;

/* Bytes of device workspace ss_fwd needs for these sizes (0 when the scan
 * runs without cross-block carries).  A pure function of its arguments. */
size_t ss_fwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype);

/*
 * Forward selective scan.
 *   u, delta      io  [Bsz, L, Dch]          required
 *   A             f32 [Dch, N]               required
 *   B, C          io  [Bsz, L, N]            required
 *   D             f32 [Dch]                  optional (NULL: no skip term)
 *   z             io  [Bsz, L, Dch]          optional (NULL: no gate)
 *   delta_bias    f32 [Dch]                  optional (NULL: no bias)
 *   softplus      nonzero: delta_eff = softplus(delta + bias); zero: delta + bias
 *   y             io  [Bsz, L, Dch]          output, required
 *   last_state    f32 [Bsz, Dch, N]          output, optional (L = 0 writes zeros)
 *   workspace     device scratch of at least ss_fwd_workspace_bytes(...) bytes
 *                 (may be NULL when that is 0); contents on entry are ignored.
 * Bsz, L or Dch equal to 0 is valid; nothing but a zero last_state is written.
 */
int ss_fwd(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
           const void *z, const float *delta_bias, int softplus, void *y, float *last_state, int64_t Bsz, int64_t L,
           int64_t Dch, int64_t N, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * ss_fwd for callers that cannot allocate device memory (no counterpart on
 * the pages this library follows; it exists for callers such as code
 * replayed from a captured CUDA graph, a custom allocator that must not be
 * bypassed, or a runtime that forbids cudaMalloc on its hot path).
 * Arguments and results are those of ss_fwd without the workspace: the
 * chunk-carry scratch lives in a library-owned device array of
 * SS_FWD_NOALLOC_MAX_SCRATCH_BYTES, reserved on every GPU that loads the
 * library until the process exits.  Problems whose ss_fwd_workspace_bytes()
 * exceeds that size are rejected with SS_ERR_WORKSPACE_TOO_SMALL before
 * anything is launched.  The function allocates nothing.  All calls share
 * the one array: calls that overlap on the GPU (unordered streams) race;
 * calls on one stream are safe.  Nothing in the array needs clearing between
 * calls.  The first call on a device that uses the scratch looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  That address is kept per
 * device ordinal for the life of the process, which assumes the runtime's one
 * primary context per device: a process that calls cudaDeviceReset on a
 * device must not call this function on it afterwards.
 */
#define SS_FWD_NOALLOC_MAX_SCRATCH_BYTES ((size_t)2 << 20)
int ss_fwd_noalloc(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
                   const void *z, const float *delta_bias, int softplus, void *y, float *last_state, int64_t Bsz,
                   int64_t L, int64_t Dch, int64_t N, int dtype, void *stream);

/*
 * Forward for training: ss_fwd that also stores, in `saved`, the states the
 * backward restarts its recomputation from, so that ss_bwd_saved can skip
 * the forward walk ss_bwd has to redo.  The pages this library follows have
 * a backward-owned record of every state (baracuda-kernels
 * `selective_scan.rs`, "Workspace": B * D * L * N elements written by the
 * backward's first pass); here the forward keeps one state in eight steps.
 *   saved         device buffer of at least ss_saved_bytes(...) bytes, 16-byte
 *                 aligned; opaque to the caller.  It receives the f32 state h
 *                 of every (b, d) row at every 8th step of L rounded up to 32
 *                 steps and, when z is given, the f32 pre-gate readout
 *                 sum_n h C + D u of every (b, t, d) (which the backward's dz
 *                 needs); without z that last part is left unwritten and
 *                 never read.
 * All other arguments and results are those of ss_fwd.  A NULL or short
 * `saved` gives SS_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 */
size_t ss_saved_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype);
int ss_fwd_save(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
                const void *z, const float *delta_bias, int softplus, void *y, float *last_state, void *saved,
                size_t saved_bytes, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, void *workspace,
                size_t workspace_bytes, void *stream);

/* Bytes of device workspace ss_bwd needs for these sizes.  A pure function
 * of its arguments. */
size_t ss_bwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype);

/*
 * Backward of the forward above for the loss sum(dy * y); the gradient
 * structure follows mamba-rs `gpu/backward.rs` (B2 gating backward, B3 SSM
 * BPTT, B4 softplus backward on the raw delta).  Inputs are the forward's
 * inputs plus dy (io, [Bsz, L, Dch]).  last_state receives no gradient.
 * Outputs, all f32 and fully overwritten:
 *   du, ddelta, dz   [Bsz, L, Dch]   (ddelta is the gradient w.r.t. the raw delta)
 *   dA               [Dch, N]        summed over batch and time
 *   dB, dC           [Bsz, L, N]     summed over channels
 *   dD, ddelta_bias  [Dch]           summed over batch and time
 * dD, dz and ddelta_bias must be given exactly when D, z and delta_bias are
 * (else SS_ERR_INVALID_PROBLEM).  The backward recomputes the forward states
 * instead of reading any saved by ss_fwd.
 *   workspace     device scratch of at least ss_bwd_workspace_bytes(...) bytes;
 *                 contents on entry are ignored.
 */
int ss_bwd(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
           const void *z, const float *delta_bias, int softplus, const void *dy, float *du, float *ddelta, float *dA,
           float *dB, float *dC, float *dD, float *dz, float *ddelta_bias, int64_t Bsz, int64_t L, int64_t Dch,
           int64_t N, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * ss_bwd reading the states ss_fwd_save stored instead of recomputing them.
 *   saved         the buffer ss_fwd_save filled for THE SAME inputs (u, delta,
 *                 A, B, delta_bias, softplus, sizes, dtype), at least
 *                 ss_saved_bytes(...) bytes; read only.  Nothing can check
 *                 that it matches: states of other inputs give the gradient
 *                 of a different forward.  NULL or short: SS_ERR_WORKSPACE_TOO_SMALL.
 *   workspace     device scratch of at least ss_bwd_saved_workspace_bytes(...)
 *                 bytes (smaller than ss_bwd's: no room for the states).
 * All other arguments and results are those of ss_bwd; the outputs are
 * bit-identical to ss_bwd's.
 */
size_t ss_bwd_saved_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype);
int ss_bwd_saved(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
                 const void *z, const float *delta_bias, int softplus, const void *dy, const void *saved,
                 size_t saved_bytes, float *du, float *ddelta, float *dA, float *dB, float *dC, float *dD, float *dz,
                 float *ddelta_bias, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Launch plan for these sizes: the largest number of time chunks a sequence
 * is cut into (ss_plan_segments gives the whole split) and how many kernels
 * each call enqueues (0 for an empty problem):
 * ss_fwd and ss_fwd_save (fwd_kernels), ss_bwd (bwd_kernels), ss_bwd_saved
 * (bwd_saved_kernels).  Pointers may be NULL.  Returns a status.
 */
int ss_plan_info(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, int64_t *chunks, int *fwd_kernels,
                 int *bwd_kernels, int *bwd_saved_kernels);

/*
 * How the launch plan splits the work.  A unit is one (batch row, tile of
 * 32 channels; 64 for N = 1); units are numbered b * ceil(Dch / tile) + tile
 * and grouped into *nseg (0 for an empty problem, else 1 or 2) consecutive
 * segments: segment i holds units[i] units, each cut into chunks[i] time
 * chunks, and every scan kernel launch covers one segment.  A second segment
 * appears when the units fill the GPU but leave a last partial round of
 * blocks (a round: 8 warps on each of its 152 SMs, 608 blocks for N >= 16):
 * those units are cut in time so that every SM gets an equal share.  The kernels of each call run in this order: the summary
 * passes of the chunked segments (in the backward followed by their carry
 * passes, which fold the reverse summaries into each chunk's incoming
 * adjoint carry), then each segment's main pass (segment 0 first), then, in
 * the backward, the two reductions.  units and chunks point
 * at 2 entries each (or NULL); nseg may be NULL.  Returns a status.
 */
int ss_plan_segments(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, int *nseg, int64_t *units,
                     int64_t *chunks);

/*
 * Measurement aid (for benchmarks).  After a call with count > 0, every
 * call of ss_fwd, ss_fwd_save, ss_fwd_ex, ss_bwd, ss_bwd_saved or ss_bwd_ex
 * made from the same host thread that returns SS_OK records events[0] on its
 * stream before its first kernel, events[i] after its i-th kernel (in the
 * order ss_plan_info counts them), stopping when the list is used up; the
 * list stays set for later calls.  events[] holds up to 16 caller-created
 * cudaEvent_t handles (passed as void*) of the calling thread's current
 * device.  count = 0 switches the recording off.  The list is per host
 * thread: calls from other threads record nothing.  Returns
 * SS_ERR_INVALID_PROBLEM for count outside 0..16 or a NULL handle.  The
 * pages this library follows have no counterpart.
 */
int ss_profile_events(void *const *events, int count);

/*
 * Extended forward: everything ss_fwd and ss_fwd_save do, plus an initial
 * state and the A_log parameterisation, through one descriptor (all fields
 * must be set; unused pointers NULL).
 *
 *   h0          f32 [Bsz, Dch, N], optional: the state before t = 0, in place
 *               of zero (the recurrence continues from it: h_0 = exp(Delta_0 A)
 *               h0 + Delta_0 B_0 u_0).  Feeding one call's last_state as the
 *               next call's h0 continues a sequence across calls (streaming
 *               prefill, sequence splits); the pages define only the zero
 *               start.
 *   a_is_log    nonzero: A holds A_log and the scan uses A = -exp(A_log)
 *               (the parameterisation mamba-rs `gpu/backward.rs` trains).
 *   saved       NULL: behaves as ss_fwd; else as ss_fwd_save (saved_bytes >=
 *               ss_saved_bytes(...)).
 * The other fields are the arguments of ss_fwd with the same meaning, layout
 * and checks; h0 must be 16-byte aligned like every pointer.  With L = 0 the
 * state stays h0: last_state receives a copy of it (zeros without h0).
 */
typedef struct {
    const void *u, *delta;    /* io [Bsz, L, Dch] */
    const float *A;           /* f32 [Dch, N]: A, or A_log when a_is_log */
    const void *B, *C;        /* io [Bsz, L, N] */
    const float *D;           /* f32 [Dch] or NULL */
    const void *z;            /* io [Bsz, L, Dch] or NULL */
    const float *delta_bias;  /* f32 [Dch] or NULL */
    const float *h0;          /* f32 [Bsz, Dch, N] or NULL */
    void *y;                  /* io [Bsz, L, Dch], output */
    float *last_state;        /* f32 [Bsz, Dch, N], output, or NULL */
    void *saved;              /* restart states for ss_bwd_ex, or NULL */
    size_t saved_bytes;
    void *workspace;          /* >= ss_fwd_workspace_bytes(...) bytes */
    size_t workspace_bytes;
    int64_t Bsz, L, Dch, N;
    int32_t dtype, softplus, a_is_log, reserved; /* reserved: set to 0 */
} ss_fwd_desc;
int ss_fwd_ex(const ss_fwd_desc *desc, void *stream);

/*
 * Extended backward: the gradient of sum(dy * y) + sum(dlast_state *
 * last_state) for the forward of ss_fwd_ex.
 *   h0, a_is_log  as in the forward.
 *   dlast_state   f32 [Bsz, Dch, N], optional: the gradient reaching
 *                 last_state from later computation (zero when NULL).
 *   dh0           f32 [Bsz, Dch, N], output: the gradient of h0, given
 *                 exactly when h0 is (else SS_ERR_INVALID_PROBLEM).  Chaining
 *                 a later segment's dh0 into the earlier segment's
 *                 dlast_state reproduces the gradients of the whole sequence.
 *   dA            with a_is_log, the gradient of A_log (dA * A).
 *   saved         NULL: recompute the states (as ss_bwd; workspace from
 *                 ss_bwd_workspace_bytes); else the buffer ss_fwd_ex filled
 *                 for the same inputs, h0 included (as ss_bwd_saved;
 *                 workspace from ss_bwd_saved_workspace_bytes).
 * The other fields are the arguments of ss_bwd with the same meaning, layout
 * and checks.  With L = 0, dh0 receives a copy of dlast_state (zeros without
 * it).  The pages this library follows have no counterpart for h0 or
 * dlast_state.
 */
typedef struct {
    const void *u, *delta;
    const float *A;
    const void *B, *C;
    const float *D;
    const void *z;
    const float *delta_bias;
    const float *h0;
    const void *dy;              /* io [Bsz, L, Dch] */
    const float *dlast_state;    /* f32 [Bsz, Dch, N] or NULL */
    const void *saved;
    size_t saved_bytes;
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *ddelta_bias;
    float *dh0;                  /* f32 [Bsz, Dch, N], iff h0 */
    void *workspace;
    size_t workspace_bytes;
    int64_t Bsz, L, Dch, N;
    int32_t dtype, softplus, a_is_log, reserved; /* reserved: set to 0 */
} ss_bwd_desc;
int ss_bwd_ex(const ss_bwd_desc *desc, void *stream);

/*
 * One recurrence step for autoregressive decoding, in place on a state kept
 * between calls (the inference use of the same recurrence; mamba-rs keeps one
 * such state per layer).  For every (b, d), with the forward's definition at
 * a single time step:
 *   state[b,d,n] <- exp(delta_eff * A[d,n]) * state[b,d,n] + delta_eff * B[b,n] * u[b,d]
 *   y[b,d]        = (sum_n state[b,d,n] * C[b,n] + D[d] * u[b,d]) * silu(z[b,d])   (new state)
 * Equivalent to ss_fwd_ex with L = 1, h0 = state and last_state = state.
 *   u, delta, z   io [Bsz, Dch] (z optional)       B, C  io [Bsz, N]
 *   A             f32 [Dch, N] (A_log when a_is_log)   D, delta_bias  f32 [Dch] optional
 *   state         f32 [Bsz, Dch, N], read and overwritten
 *   y             io [Bsz, Dch], output
 * Checks as ss_fwd (sizes, N in {1,2,4,8,16,32}, required pointers, 16-byte
 * alignment).  One kernel, no workspace.  The pages this library follows have
 * no single-step entry point.
 */
int ss_decode_step(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
                   const void *z, const float *delta_bias, int softplus, int a_is_log, float *state, void *y,
                   int64_t Bsz, int64_t Dch, int64_t N, int dtype, void *stream);

/* Device-side failures.  The scan kernels stage their tiles into shared
 * memory with TMA copies (cp.async.bulk.tensor) that complete on an mbarrier;
 * a copy lands within microseconds, and every wait on one gives up after two
 * seconds.  A block that gives up leaves SS_ERR_DEVICE_TIMEOUT in the
 * library's device status word (one per device, shared by all calls), waits
 * once more (bounded) for its own copies and returns, so the context stays
 * usable; the outputs of that call are then incomplete.  A launch returns
 * before its kernels run, so this failure is not part of the calls' return
 * codes.
 *
 * A block also checks, before its first copy, that its shared-memory tile
 * buffers have the 128-byte alignment TMA boxes need; if not (not expected:
 * they are declared so), it stages with per-thread copies and notes that in
 * the status word.
 *
 * ss_device_status: waits for `stream` (the current device's), reads the
 * status word and clears it.  SS_OK when nothing was noted since the last
 * read; SS_ERR_DEVICE_TIMEOUT when a kernel gave up waiting (this wins over
 * the next); SS_ERR_STAGING_FALLBACK when a kernel staged without TMA;
 * SS_ERR_CUDA when the read failed.  Kernels on other streams still running
 * are not waited for.
 */
int ss_device_status(void *stream);

/* Runs one block on `stream` that waits on a barrier nothing completes, for
 * limit_ns nanoseconds (0 .. 2e9; else SS_ERR_INVALID_PROBLEM), then reports
 * the wait as failed in the status word exactly as a scan kernel does.  For
 * testing the status path without any failure of the GPU.  Returns the
 * launch's status; read the outcome with ss_device_status.
 */
int ss_selftest_wait_timeout(int64_t limit_ns, void *stream);

/* Staging choice for the following calls of the process: 0 (the default)
 * uses TMA wherever the problem allows it (D and N times the element size
 * multiples of 16 bytes, D a multiple of 4), 1 stages every tile with
 * per-thread asynchronous copies instead.  Both produce identical results;
 * the switch exists to test that.  Returns the previous setting.  Not ordered
 * against calls running on other host threads.
 */
int ss_set_copies_only(int enable);

/* 1 when the scan kernels of a problem of these sizes stage their tiles with
 * TMA under the current setting of ss_set_copies_only, else 0 (also for
 * invalid or empty problems, and where the driver offers no tensor-map
 * encoder).  Touches no device memory. */
int ss_staging_uses_tma(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype);

/* Throughput of the GPU's exponential unit: MUFU ex2.approx.f32 results per
 * SM clock cycle per SM on the current device, measured by one block per SM
 * running `iters` rounds of eight independent exponential chains per thread
 * (1 .. 2^20; about 0.5 ms at 4096), each block timed by its SM's cycle
 * counter; the median over the SMs.  This is the peak of the scan's
 * exponential roofline (one 2^x per (t, d, n) and direction).  Synchronous;
 * allocates and frees a few bytes of device memory.
 */
int ss_measure_ex2_rate(int iters, double *per_clk_per_sm);

/* Throughput of the GPU's FP32 pipe: f32 results of fused multiply-adds per
 * SM clock cycle per SM on the current device, measured like
 * ss_measure_ex2_rate with eight independent chains of packed f32x2 FMAs per
 * thread (each two results; the form the scan kernels issue their
 * multiplies and multiply-adds in).  This is the peak of the scan's FP32
 * roofline: every f32 multiply, add or multiply-add of a state update takes
 * one such result slot.  Same arguments, errors and side effects as
 * ss_measure_ex2_rate.
 */
int ss_measure_fma_rate(int iters, double *per_clk_per_sm);

/* Static description of a status code. */
const char *ss_status_string(int status);

/* ABI version (2: ss_fwd_save / ss_bwd_saved added, ss_plan_info gained
 * bwd_saved_kernels; 3: ss_fwd_ex / ss_bwd_ex / ss_decode_step added; 4:
 * ss_plan_segments added, the saved-state buffer sized by L rounded up to 32
 * steps; 5: a saved state every 8 steps, ss_device_status /
 * ss_selftest_wait_timeout / ss_set_copies_only added; 6: the saved states
 * of ss_fwd_save laid out by (batch row, channel tile) then time and
 * interleaved by channel within a block (a buffer written by an earlier
 * version is not read correctly), ss_measure_fma_rate added; 7: in the
 * backward a chunked segment runs a carry pass between its reverse summaries
 * and its main pass, which ss_plan_info counts and ss_profile_events marks);
 * bumped on any incompatible change. */
int ss_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SS_H */

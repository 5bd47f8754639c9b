/*
 * lrscan.h -- C ABI of the GB300 (sm_103a) gated linear-recurrence scan
 * library.  Forward-only; one GPU; the kernels are hand-written CUDA.
 *
 * Every scan computes a recurrence  h_t = a_t (.) h_{t-1} + b_t  with a
 * readout, over post-projection, post-activation inputs, starting from an
 * optional initial state and returning the outputs and the final state.
 *
 * Sources (web pages, cited by title and section):
 *   [SSM]   cortexnet 3.2.1 wheel, cortexnet/ssm.py -- module docstring (ZOH
 *           discretisation), MultiScaleSSM.__init__ (multi-scale A_log, D),
 *           MultiScaleSSM.forward (A = -exp(A_log), dt = softplus(dt_proj(x)),
 *           D skip, silu(z) gate, past_state / new_state),
 *           MultiScaleSSM._selective_scan (the recurrence, in float32).
 *   [RGLRU] lrnnx docs, lrnnx.models.ltv.rglru module source -- RGLRU.forward
 *           (gates, rglru_scan_fn(u, delta, a, return_last_state)) and
 *           RGLRU.step (fallback update a^(c r), sqrt(1 - a^2)).
 *   [HGRN2] frankenstein-transformer docs, HGRN2 Attention page --
 *           S_t = diag(g_t) S_{t-1} + v_t k_t^T, per-head matrix state,
 *           lower-bounded forget gate, hidden % heads check.
 *   [MINMAX] minmaxrnc 0.1.0 wheel -- minmax_neuron.py (MinMaxNeuron:
 *           x_{t+1} = max(min(r_t, x_t), s_t), forward returns every state
 *           and the last one), minmax_operator.py (apply, compose).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or retains them.  Every tensor is dense and
 *    row-major (last index fastest) in the layout written beside it.  A
 *    required pointer may be NULL only when its tensor has no elements.
 *  - Each tensor's base address must be 16-byte aligned (LR_ERR_MISALIGNED).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are returned synchronously and launch
 *    nothing.  A failed launch returns LR_ERR_CUDA.
 *  - Errors detected on the device (a bounded wait that ran out, an HGRN2
 *    gate that is not a number) are recorded per call: the first 256 bytes
 *    of the call's workspace hold its status word, stamped with the call, so
 *    the word always describes the latest call that used the workspace.
 *    lr_check_status(workspace, stream) reads and resets it.
 *  - State and arithmetic are float32 whatever the I/O dtype; bf16 outputs
 *    are rounded once, at the store.  There is no CPU fallback.
 *  - `workspace` is caller-owned device scratch of at least the size the
 *    matching *_workspace_size() call returns for the same sizes on the
 *    current device: always at least 256 bytes (the status), also for an
 *    empty problem; 0 means the arguments are invalid.  Its contents need no
 *    initialisation.  Calls that overlap in time must use distinct
 *    workspaces.
 *  - The setters under "Tuning and test hooks" change process-wide settings
 *    read at each call's launch; they are not synchronised with calls
 *    running on other host threads.
 */
#ifndef LRSCAN_H
#define LRSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA
 * headers. */
typedef struct CUstream_st *lr_stream_t;

/* I/O element type of the activation tensors. */
typedef enum { LR_F32 = 0, LR_BF16 = 1 } lr_dtype;

/* Status codes (0 = success, negative = error). */
enum {
    LR_OK = 0,
    LR_ERR_INVALID_ARG = -1,  /* NULL required pointer, negative size, bad scalar */
    LR_ERR_UNSUPPORTED = -2,  /* legal but unsupported shape or dtype */
    LR_ERR_MISALIGNED = -3,   /* a tensor base is not 16-byte aligned */
    LR_ERR_WORKSPACE = -4,    /* workspace NULL or smaller than required */
    LR_ERR_CUDA = -5,         /* a CUDA runtime/driver call failed */
    LR_ERR_TIMEOUT = -6,      /* device side: a bounded wait ran out */
    LR_ERR_RANGE = -7         /* device side: an HGRN2 gate that is not a finite number */
};

/* Human-readable name of a status code (static storage). */
const char *lr_status_string(int code);

/* Library version, major*10000 + minor*100 + patch. */
int lr_version(void);

/*
 * Device-side status of the latest call that used `workspace`.
 *
 * Every call that takes a workspace keeps its device-side status in the
 * workspace's first 256 bytes: each call stamps them afresh, so they describe
 * that call alone, whatever the memory held before (no initialisation is
 * needed).  lr_check_status synchronises `stream` -- the stream the call was
 * made on -- then returns the status recorded there (LR_OK, or e.g.
 * LR_ERR_TIMEOUT when a bounded wait of that call ran out; the call's
 * outputs are then not meaningful) and resets it to LR_OK.  Concurrent calls
 * on different streams with distinct workspaces are checked independently.
 * workspace == NULL reads the status of the latest
 * lr_rglru_scan_fwd_noalloc call on the current device (kept in that entry
 * point's built-in scratch).  Returns LR_ERR_CUDA if a CUDA call fails.
 */
int lr_check_status(void *workspace, lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Selective SSM scan                                                        */
/* ------------------------------------------------------------------------ */

/*
 * [SSM] MultiScaleSSM._selective_scan + the D skip and silu(z) gate of
 * MultiScaleSSM.forward.  For every batch b and channel d, with the state
 * h[n] = h0[b,d,n] (zero when h0 == NULL) and A[n] = -exp(A_log[d,n]):
 *
 *   delta_t = dt_softplus ? softplus(dt[b,t,d]) : dt[b,t,d]
 *             (softplus as torch: identity above 20, else log(1 + e^x))
 *   h[n]    = exp(delta_t * A[n]) * h[n] + delta_t * Bm[b,t,n] * x[b,t,d]
 *   y[b,t,d] = (sum_n Cm[b,t,n] h[n] + Dskip[d] x[b,t,d]) * silu(z[b,t,d])
 *
 * and h_final[b,d,:] = h after the last step.  The readout uses the state
 * after the update at t.  B_t and C_t are shared by all channels.
 *
 * Decays: where A_log sits on the multi-scale initialisation lattice
 * (MultiScaleSSM.__init__: A[n] = (n+1) A[0], to 2^-20 relative in fp32 for
 * every state of the 64 channels a warp holds, which the kernel checks
 * itself) the 16 decays of a step are computed as powers of exp(delta A[0]);
 * elsewhere as one exp per state.  The two forms differ by rounding only
 * (well inside max|y - y_exact| <= 1e-4 max|y_exact| for fp32 I/O and 1e-2
 * for bf16 I/O); the caller chooses nothing.
 *
 * Parallel pieces: the kernel cuts each sequence into pieces that run in
 * parallel.  A piece that starts inside the sequence rebuilds its starting
 * state from the preceding steps back to where the carried state has decayed
 * below 2^-10 (bf16 I/O) or 2^-32 (fp32 I/O) of its size, or takes it from
 * the preceding pieces (see lr_set_selective_warmup); the history left out
 * is below that share, inside the tolerances above.  Results therefore
 * depend on the rounding of the piece boundaries, which depend on the
 * device's SM count and on B, L, D.
 *
 * Layouts: x, dt, z, y: (B, L, D) in `io`; Bm, Cm: (B, L, N) in `io`;
 *          A_log: (D, N) fp32; Dskip: (D) fp32; h0, h_final: (B, D, N) fp32.
 * Optional (NULL allowed): z (no gate), Dskip (no skip), h0 (zero state),
 *          h_final (not written).
 * Requirements: N == 16; D % 8 == 0 (bf16) or D % 4 == 0 (fp32), else
 *          LR_ERR_UNSUPPORTED; delta >= 0 (a step size; with dt_softplus it
 *          always is).  B, L may be 0 (nothing is launched; h_final = h0).
 */
size_t lr_selective_scan_workspace_size(int64_t B, int64_t L, int64_t D,
                                        int64_t N, lr_dtype io);

int lr_selective_scan_fwd(const void *x, const void *dt, const void *z,
                          const void *Bm, const void *Cm,
                          const float *A_log, const float *Dskip,
                          const float *h0, void *y, float *h_final,
                          int64_t B, int64_t L, int64_t D, int64_t N,
                          lr_dtype io, int dt_softplus,
                          void *workspace, size_t ws_bytes, lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* RG-LRU scalar-state scan                                                  */
/* ------------------------------------------------------------------------ */

/*
 * [RGLRU] RGLRU.step fallback update applied at every step (the scan that
 * rglru_scan_fn performs in RGLRU.forward).  For every b and channel d, with
 * h = h0[b,d] (zero when NULL):
 *
 *   a_t = exp(c * r[b,t,d] * a_log[d])        (= a^(c r) with a = exp(a_log))
 *   h   = a_t * h + sqrt(1 - a_t^2) * (i[b,t,d] * x[b,t,d])
 *   y[b,t,d] = h
 *
 * and h_final[b,d] = h after the last step.  r and i are the recurrent and
 * input gates after their sigmoid; c is the fixed gate scale (8 on the page).
 *
 * Layouts: x, r, i, y: (B, L, D) in `io`; a_log: (D) fp32 (<= 0);
 *          h0, h_final: (B, D) fp32.  Optional: h0, h_final.
 * Requirements: D % 8 == 0 (bf16) or D % 4 == 0 (fp32), else
 *          LR_ERR_UNSUPPORTED; c finite.
 */
size_t lr_rglru_scan_workspace_size(int64_t B, int64_t L, int64_t D,
                                    lr_dtype io);

int lr_rglru_scan_fwd(const void *x, const void *r, const void *i,
                      const float *a_log, float c, const float *h0,
                      void *y, float *h_final,
                      int64_t B, int64_t L, int64_t D, lr_dtype io,
                      void *workspace, size_t ws_bytes, lr_stream_t stream);

/*
 * RG-LRU scan for callers that cannot allocate device memory.  The source
 * pages have no counterpart; this entry point exists for the library's
 * users.  Some host frameworks and runtimes own every byte of device memory
 * through their own allocator or fix their memory budget at start-up, and
 * some latency-critical paths cannot afford cudaMalloc's implicit device
 * synchronisation; such callers have no way to provide the workspace that
 * lr_rglru_scan_fwd may need.
 *
 * Same arguments, arithmetic, layouts and results as lr_rglru_scan_fwd, minus
 * the workspace: the look-back scratch comes from a fixed array of 1 MiB
 * (1048576 bytes) built into the library, which every GPU that loads the
 * library holds until the process exits.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - A problem whose look-back state would exceed 1 MiB is rejected with
 *     LR_ERR_WORKSPACE before anything is launched (automatic splitting never
 *     needs more than about 0.4 MiB; only a large lr_set_split_override can).
 *   - All calls on a device share the array and it keeps the previous call's
 *     contents; each call clears the part that must start at zero.  Calls
 *     that overlap in time on the GPU (different streams) race on it and must
 *     be serialised by the caller.
 */
int lr_rglru_scan_fwd_noalloc(const void *x, const void *r, const void *i,
                              const float *a_log, float c, const float *h0,
                              void *y, float *h_final,
                              int64_t B, int64_t L, int64_t D, lr_dtype io,
                              lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* HGRN2 matrix-state recurrence                                             */
/* ------------------------------------------------------------------------ */

/*
 * [HGRN2] HGRN2Attention: per batch b and head h a dv x dk state S (row i =
 * value channel, column j = key channel), S = S0[b,h] (zero when NULL):
 *
 *   S_t = diag(g_t) S_{t-1} + v_t k_t^T        (g_t scales the rows of S)
 *   o_t = S_t q_t                              (after the update at t)
 *
 * and S_final[b,h] = S after the last step.  g is the forget gate after its
 * activation and lower bound, in [0, 1].
 *
 * Layouts: q, k: (B, L, H*dk); v, g, o: (B, L, H*dv), all in `io`;
 *          S0, S_final: (B, H, dv, dk) fp32.  Optional: S0, S_final.
 * Requirements: H > 0, dk >= 1, dv >= 1, chunk >= 1; dk <= 512 (else
 *          LR_ERR_UNSUPPORTED).
 * Two kernels: dk == dv == 128 with chunk == 64 and bf16 I/O runs the
 *          chunked tcgen05 tensor-core kernel; every other shape or fp32 I/O
 *          runs a step-by-step CUDA-core kernel (fp32 arithmetic throughout,
 *          O(L dk dv) work, no gate-range limit; `chunk` is not used there).
 *          On the tensor-core path every gate in [0, 1] is handled: a
 *          chunk whose gates decay too steeply for its factorisation is run in
 *          shorter pieces, and a gate below 2^-120 (0 included) acts as a
 *          reset of that state row.  The call is two launches: the first runs
 *          every chunk whole and marks the thread blocks (64 value channels
 *          of one batch row and head) that met a steep chunk; the second
 *          re-runs only those, in pieces (it returns at once when none was
 *          marked, and is not launched by lr_hgrn2_preact_fwd when
 *          lb >= 0.18, which rules steep chunks out).  A gate that is not a finite number sets
 *          LR_ERR_RANGE (read with lr_check_status); that call's outputs are
 *          then not meaningful.  Gates above 1 lie outside the recurrence's
 *          domain and give undefined results.
 * Workspace: lr_hgrn2_workspace_size bytes: the call's device status and,
 *          on the tensor-core path, one 8-byte mark per thread block
 *          (B * H * 2).
 */
size_t lr_hgrn2_workspace_size(int64_t B, int64_t L, int64_t H, int64_t dk,
                               int64_t dv, lr_dtype io);

int lr_hgrn2_fwd(const void *q, const void *k, const void *v, const void *g,
                 const float *S0, void *o, float *S_final,
                 int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                 int64_t chunk, lr_dtype io,
                 void *workspace, size_t ws_bytes, lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Gates given before their activation                                       */
/* ------------------------------------------------------------------------ */

/*
 * The pages activate the gates right before their scans: [RGLRU] forward
 * applies sigmoid to the r and i projections, [HGRN2] lower-bounds a
 * sigmoid-activated forget gate, g = lb + (1 - lb) sigmoid(f).  These entry
 * points take the pre-activation tensors and apply the activation inside the
 * scan kernel, so callers need no separate elementwise pass; otherwise they
 * are lr_rglru_scan_fwd and lr_hgrn2_fwd (same layouts, requirements,
 * workspace and errors).  lr_hgrn2_preact_fwd: lb in [0, 1) (else
 * LR_ERR_INVALID_ARG); f is (B, L, H*dv) like g.
 */
int lr_rglru_scan_preact_fwd(const void *x, const void *r_pre, const void *i_pre,
                             const float *a_log, float c, const float *h0,
                             void *y, float *h_final,
                             int64_t B, int64_t L, int64_t D, lr_dtype io,
                             void *workspace, size_t ws_bytes, lr_stream_t stream);

int lr_hgrn2_preact_fwd(const void *q, const void *k, const void *v, const void *f,
                        float lb, const float *S0, void *o, float *S_final,
                        int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                        int64_t chunk, lr_dtype io,
                        void *workspace, size_t ws_bytes, lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MinMax recurrence                                                         */
/* ------------------------------------------------------------------------ */

/*
 * [MINMAX] MinMaxNeuron: for every batch row b and channel d,
 *
 *   x_t = max(min(r_t, x_{t-1}), s_t),   y_t = x_t   (the state after step t)
 *
 * with x_{-1} = x0[b,d] (zero when x0 == NULL, the neuron's default initial
 * state) and x_final[b,d] = x after the last step.  r and s are the outputs
 * of the neuron's two projections.  min and max select one argument, so the
 * result is exact (every y equals an input or x0, rounded to `io` at the
 * store only when x0 is not representable in it); a NaN argument gives NaN
 * from then on, as torch.minimum / torch.maximum in the page's apply.
 *
 * Layouts: r, s, y: (B, L, D) in `io`; x0, x_final: (B, D) fp32.
 * Optional: x0, x_final.
 * Requirements: D % 8 == 0 for bf16, D % 4 == 0 for fp32 (LR_ERR_UNSUPPORTED).
 * Workspace: as for the other diagonal scans (look-back scratch when the
 * library splits time; query lr_minmax_scan_workspace_size).
 */
size_t lr_minmax_scan_workspace_size(int64_t B, int64_t L, int64_t D, lr_dtype io);

int lr_minmax_scan_fwd(const void *r, const void *s, const float *x0, void *y,
                       float *x_final, int64_t B, int64_t L, int64_t D, lr_dtype io,
                       void *workspace, size_t ws_bytes, lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Host buffers                                                              */
/* ------------------------------------------------------------------------ */

/*
 * The scans above with every tensor in HOST memory (activations, parameters,
 * initial and final states); only the workspace is device memory, on the
 * current device.  The pages' layers take their inputs from wherever the
 * framework keeps them; these entry points are for callers whose data lives
 * in host memory, so that the host <-> device traffic, which dominates such a
 * call, overlaps the scan.
 *
 * The library cuts the sequence into chunks of Lc time steps (a multiple of
 * 64, about 128 MB of inputs each) and runs each chunk with the matching
 * device entry point, the state carried from chunk to chunk on the device;
 * on three streams of its own it copies chunk k+1's inputs in while chunk k
 * runs and chunk k-1's outputs go out.  Arguments, layouts, requirements and
 * errors are those of the device call (lr_selective_scan_fwd,
 * lr_rglru_scan_fwd, lr_hgrn2_fwd, lr_minmax_scan_fwd); results equal the
 * device call's up to the rounding of the chunk boundaries (the same
 * split-resume property that h0 / h_final give).
 *
 *   - Ownership: every host pointer stays the caller's; the call reads and
 *     writes them until it returns, and it returns only when every output
 *     and the final state are in host memory.  Work already queued on
 *     `stream` completes before the library touches the workspace.
 *   - Pinned (page-locked) host memory lets the copies run asynchronously
 *     and overlap; pageable memory gives the same results, slower.
 *   - workspace: at least lr_*_fwd_host_workspace_size(...) bytes of device
 *     memory, 16-byte aligned, else LR_ERR_WORKSPACE / LR_ERR_MISALIGNED
 *     (two chunks of inputs and of outputs, two states, the parameters and
 *     the device call's own workspace).  The size covers the optional
 *     tensors (z, Dskip) whether or not a call passes them.
 *   - Calls on one device run one after another (the library's streams are
 *     shared; a mutex serialises them).  The *_async forms below queue the
 *     same work and return without waiting for it.
 */
size_t lr_selective_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D,
                                                 int64_t N, lr_dtype io);
int lr_selective_scan_fwd_host(const void *x, const void *dt, const void *z,
                               const void *Bm, const void *Cm,
                               const float *A_log, const float *Dskip,
                               const float *h0, void *y, float *h_final,
                               int64_t B, int64_t L, int64_t D, int64_t N,
                               lr_dtype io, int dt_softplus,
                               void *workspace, size_t ws_bytes, lr_stream_t stream);

size_t lr_rglru_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D,
                                             lr_dtype io);
int lr_rglru_scan_fwd_host(const void *x, const void *r, const void *i,
                           const float *a_log, float c, const float *h0,
                           void *y, float *h_final,
                           int64_t B, int64_t L, int64_t D, lr_dtype io,
                           void *workspace, size_t ws_bytes, lr_stream_t stream);

size_t lr_hgrn2_fwd_host_workspace_size(int64_t B, int64_t L, int64_t H, int64_t dk,
                                        int64_t dv, lr_dtype io);
int lr_hgrn2_fwd_host(const void *q, const void *k, const void *v, const void *g,
                      const float *S0, void *o, float *S_final,
                      int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                      int64_t chunk, lr_dtype io,
                      void *workspace, size_t ws_bytes, lr_stream_t stream);

size_t lr_minmax_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D,
                                              lr_dtype io);
int lr_minmax_scan_fwd_host(const void *r, const void *s, const float *x0, void *y,
                            float *x_final, int64_t B, int64_t L, int64_t D,
                            lr_dtype io, void *workspace, size_t ws_bytes,
                            lr_stream_t stream);

/*
 * Asynchronous forms of the four host-buffer calls (a library facility; the
 * pages specify only the recurrences).  Same arguments, checks and results
 * as the synchronous forms, but each returns once its chunks are queued on
 * the library's streams, so consecutive calls overlap: the next call's
 * inputs go in while this call's last chunks run and its outputs come out.
 *   - Every host buffer of the call stays in use (inputs read, outputs and
 *     the final state written) until lr_host_sync() returns: the caller keeps
 *     them allocated and unchanged and reads no result before then.
 *   - Each call in flight needs a workspace of its own (two calls sharing one
 *     would overwrite each other's staging buffers); it too is in use until
 *     lr_host_sync() returns.
 *   - A call must not read a host buffer that an earlier call in flight
 *     writes (running a sequence in segments through h_final -> h0 needs
 *     lr_host_sync() between the segments).
 *   - Errors found before anything is queued (arguments, workspace size)
 *     are returned as by the synchronous form.  The device-side status of a
 *     call (a bounded wait that ran out) is read after lr_host_sync() with
 *     lr_check_status(workspace, stream).
 * Calls on one device queue in call order (a mutex serialises the queueing).
 */
int lr_selective_scan_fwd_host_async(const void *x, const void *dt, const void *z,
                                     const void *Bm, const void *Cm,
                                     const float *A_log, const float *Dskip,
                                     const float *h0, void *y, float *h_final,
                                     int64_t B, int64_t L, int64_t D, int64_t N,
                                     lr_dtype io, int dt_softplus,
                                     void *workspace, size_t ws_bytes, lr_stream_t stream);
int lr_rglru_scan_fwd_host_async(const void *x, const void *r, const void *i,
                                 const float *a_log, float c, const float *h0,
                                 void *y, float *h_final,
                                 int64_t B, int64_t L, int64_t D, lr_dtype io,
                                 void *workspace, size_t ws_bytes, lr_stream_t stream);
int lr_hgrn2_fwd_host_async(const void *q, const void *k, const void *v, const void *g,
                            const float *S0, void *o, float *S_final,
                            int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                            int64_t chunk, lr_dtype io,
                            void *workspace, size_t ws_bytes, lr_stream_t stream);
int lr_minmax_scan_fwd_host_async(const void *r, const void *s, const float *x0, void *y,
                                  float *x_final, int64_t B, int64_t L, int64_t D,
                                  lr_dtype io, void *workspace, size_t ws_bytes,
                                  lr_stream_t stream);

/*
 * Waits until every host-buffer call queued on the current device has
 * finished (its outputs and final state are in host memory).  Returns LR_OK,
 * or LR_ERR_CUDA when a CUDA call failed.
 */
int lr_host_sync(void);

/* ------------------------------------------------------------------------ */
/* Single-token decode steps                                                 */
/* ------------------------------------------------------------------------ */

/*
 * One step (L = 1) of each recurrence with a carried state, as the pages run
 * their layers token by token:
 *   [SSM] MultiScaleSSM.forward with past_state and one token,
 *   [RGLRU] RGLRU.step, [HGRN2] the per-token update S = diag(g) S + v k^T.
 * The arithmetic is that of the matching *_fwd call with L = 1 (same inputs,
 * same readout after the update); the kernels use the accurate math library
 * functions.  The state before the step (h_in / S_in) may be NULL for a zero
 * state; the state after it (h_out / S_out) is always written and may be the
 * same buffer as h_in / S_in (in-place update).  No workspace.  Shapes:
 *   selective: x, dt, z, y: (B, D) io; Bm, Cm: (B, N) io; A_log: (D, N) fp32;
 *              Dskip: (D) fp32 or NULL; z NULL = no gate; h_in, h_out:
 *              (B, D, N) fp32.  N must be 16.
 *   rglru:     x, r, i, y: (B, D) io; a_log: (D) fp32; h_in, h_out: (B, D)
 *              fp32.
 *   hgrn2:     q, k: (B, H*dk) io; v, g, o: (B, H*dv) io; S_in, S_out:
 *              (B, H, dv, dk) fp32.  Any dk, dv >= 1 and either io dtype.
 * Errors: LR_ERR_INVALID_ARG for a NULL required pointer or a negative size,
 * LR_ERR_UNSUPPORTED for N != 16, LR_ERR_MISALIGNED as for every call.
 */
int lr_selective_scan_step(const void *x, const void *dt, const void *z,
                           const void *Bm, const void *Cm,
                           const float *A_log, const float *Dskip,
                           const float *h_in, float *h_out, void *y,
                           int64_t B, int64_t D, int64_t N, lr_dtype io,
                           int dt_softplus, lr_stream_t stream);

int lr_rglru_scan_step(const void *x, const void *r, const void *i,
                       const float *a_log, float c, const float *h_in,
                       float *h_out, void *y, int64_t B, int64_t D,
                       lr_dtype io, lr_stream_t stream);

/* MinMax ([MINMAX] MinMaxNeuron, one token): x = max(min(r, x), s), y = x.
 * r, s, y: (B, D) io; x_in (NULL = zero), x_out: (B, D) fp32. */
int lr_minmax_scan_step(const void *r, const void *s, const float *x_in,
                        float *x_out, void *y, int64_t B, int64_t D, lr_dtype io,
                        lr_stream_t stream);

int lr_hgrn2_step(const void *q, const void *k, const void *v, const void *g,
                  const float *S_in, float *S_out, void *o,
                  int64_t B, int64_t H, int64_t dk, int64_t dv, lr_dtype io,
                  lr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Tuning and test hooks                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Overrides the number of time splits the two diagonal scans use (0 =
 * automatic).  With more than one split, consecutive time ranges of a
 * channel block run in different thread blocks that pass their carries by a
 * decoupled look-back; workspace sizes follow the override.  Process-wide,
 * not thread-safe.  Returns the previous value.
 */
int lr_set_split_override(int splits);

/*
 * Tuning / test knob of the selective scan.  The kernel cuts sequences into
 * pieces that run in parallel.  A piece that starts inside a sequence first
 * rebuilds the state reached just before it from the preceding steps, back
 * to where every channel's slowest decay has fallen below 2^-10 (bf16 I/O) or
 * 2^-32 (fp32 I/O), so that the history left out contributes less than that
 * share of the state's size (a "warm-up"), when that window lies within
 * `max_steps` steps; otherwise it runs from zero, takes its carry from the
 * preceding pieces by decoupled look-back and corrects its outputs by the
 * carry's contribution (to the same cut-off).  With warm-ups on, a warp
 * that has run out of work splits off the back half of the largest range
 * still unclaimed and warms up to its start (so results can differ between
 * runs within the cut-off).  0 disables the warm-up (every carry by
 * look-back, a fixed partition); a negative value restores the automatic
 * setting: 2048 steps for bf16 I/O, 0 for fp32 I/O (whose 2^-32 window is
 * about as long as the pages' sequences).  Process-wide, not thread-safe.
 * Returns the previous setting (-1: automatic).
 */
int64_t lr_set_selective_warmup(int64_t max_steps);

/*
 * Tuning / test knob: the chunk length (time steps) of the host-buffer entry
 * points (lr_*_fwd_host); 0 restores the automatic choice (a multiple of 64
 * steps holding about 128 MB of inputs).  Any positive length is valid: chunk
 * boundaries need not fall on a kernel tile.  Process-wide; set it before
 * querying a host workspace size, which depends on it.  Returns the previous
 * setting.
 */
int64_t lr_set_host_chunk_steps(int64_t steps);

/*
 * Test hook for the bounded look-back wait: when `split` >= 1, the thread
 * blocks of that time split never publish their carries, so their successors'
 * waits run out (after about `timeout_ms` milliseconds), set LR_ERR_TIMEOUT
 * and finish with a zero carry.  -1 disables.  Process-wide, not
 * thread-safe.  Returns LR_OK.
 */
int lr_test_withhold_split(int split, int timeout_ms);

#ifdef __cplusplus
}
#endif

#endif /* LRSCAN_H */

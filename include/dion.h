/*
 * dion.h -- C ABI of libdion: the orthonormalized optimizer step on one GPU
 * (NVIDIA GB300, sm_103a).
 *
 * Two operations, each applied to a megabatch of same-shape weight matrices
 * ("microsoft/dion" repository summary: parameters of one shape are grouped
 * and processed as one batch; project card, "How it works": parameters are
 * processed in batches):
 *
 *   dion_step_batched  the legacy Dion update: amortized power iteration with
 *                      error feedback at a low rank r ("Dion: The distributed
 *                      orthonormal update revolution is here", the Dion and
 *                      low-rank-fraction paragraphs; "Dion: Distributed
 *                      Orthonormalized Updates", abstract).  Per matrix:
 *                        B = M + G
 *                        P = orthonormalize(B Q)             (m x r)
 *                        R = B^T P                            (n x r)
 *                        M <- B - (1 - mu) P R^T              (error feedback)
 *                        Q <- R with unit-norm columns
 *                        X <- (1 - lr*wd) X - lr*sqrt(m/n) P Q^T
 *   muon_ns_batched    Muon: Newton-Schulz orthogonalization of the (momentum
 *                      of the) gradient, whole-matrix or per attention head
 *                      (talk page, orthonormal-update paragraph; project card,
 *                      "Highlights": per-head Newton-Schulz).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major batched
 *     tensors; matrix k of a [batch, rows, cols] tensor starts at element
 *     k*rows*cols.  Base pointers must be 16-byte aligned.
 *   - The caller owns all memory, including the workspace, whose size the
 *     *_workspace_size functions give.  The library never allocates, frees
 *     or synchronizes: it enqueues kernels on `cuda_stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and returns.
 *   - Argument errors (shape, null pointer, alignment, dtype, workspace too
 *     small) are detected on the host and returned before anything is
 *     enqueued.  A failed kernel launch returns DION_ERR_CUDA.
 *   - Numeric events found on the device do not trap: they are recorded in a
 *     status word inside the workspace, read with dion_get_status after the
 *     caller has synchronized the stream (bits listed there).  A column of
 *     P whose part outside the span of the columns before it is below 1e-6
 *     of its norm (P rank deficient to that tolerance, decided in float64)
 *     is set to zero, so the step still completes with finite output at a
 *     lower rank.
 *   - Calls are not thread-safe with respect to one workspace: two calls in
 *     flight at once must use different workspaces.
 */
#ifndef DION_H
#define DION_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DION_OK = 0,
    DION_ERR_INVALID_ARG = 1,   /* bad shape, rank, null pointer or alignment */
    DION_ERR_UNSUPPORTED = 2,   /* valid request this build does not handle */
    DION_ERR_WORKSPACE = 3,     /* workspace pointer NULL or too small */
    DION_ERR_CUDA = 4,          /* a CUDA call or kernel launch failed */
    DION_ERR_NUMERIC = 5        /* device-side numeric breakdown (see above) */
} dion_status;

typedef enum {
    DION_F32 = 0,               /* X and G (and O) are float32 */
    DION_BF16 = 1               /* X and G (and O) are bfloat16 */
} dion_dtype;                   /* M, Q are always float32 */

/*
 * Workspace bytes needed by dion_step_batched for this shape.
 * Returns DION_ERR_INVALID_ARG unless batch >= 1, m, n >= 1, 1 <= r <= min(m, n)
 * and bytes != NULL.
 */
dion_status dion_workspace_size(int batch, int m, int n, int r, dion_dtype dt, size_t* bytes);

/*
 * One Dion step on `batch` matrices of shape m x n at rank r.
 *   X  [batch, m, n] dt      weights, updated in place
 *   G  [batch, m, n] dt      gradients, read only
 *   M  [batch, m, n] float   momentum buffers, updated in place
 *   Q  [batch, n, r] float   right factors, updated in place; the caller
 *                            supplies the initial Q (any full-rank Q, e.g.
 *                            Gaussian with unit-norm columns)
 *   mu                       error-feedback momentum (0 <= mu <= 1)
 *   lr, weight_decay         X <- (1 - lr*weight_decay) X - lr*sqrt(m/n) P Q^T
 *   workspace                >= dion_workspace_size(...) bytes, device memory,
 *                            256-byte aligned; its contents need not be
 *                            initialized and are scratch after the call
 *                            (except the status word, see dion_get_status)
 * P is orthonormalized by CholeskyQR2 in float32.  Matrices whose first
 * float32 pass meets a pivot below 1e-6 of its column's squared norm (a
 * dominant direction: P's condition number beyond about 1e3, or true rank
 * deficiency) redo that first pass in float64 from the same panel, which
 * resolves condition numbers up to about 1e7; the other matrices of the
 * batch are not affected.  That fallback costs O(r^3) float64 work on one SM
 * per flagged matrix (about 0.1 s at r = 1024).
 */
dion_status dion_step_batched(int batch, int m, int n, int r, dion_dtype dt,
                              void* X, const void* G, float* M, float* Q,
                              float mu, float lr, float weight_decay,
                              void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * dion_step_batched with mu, lr and weight_decay read on the device, when the
 * step's kernels run, from hyper[0], hyper[1], hyper[2] (three float32 values
 * in device memory, 4-byte aligned, owned by the caller).  The step enqueues
 * only kernels and asynchronous memsets on cuda_stream, allocates nothing and
 * never synchronizes, so it can be captured in a CUDA graph once and replayed
 * every step while the caller writes the schedule's values into hyper (with
 * any stream-ordered copy) between replays; the same shapes, pointers and
 * workspace are used by every replay.  The first call for a shape should be
 * made outside a capture (it sets per-kernel launch attributes once).
 * Both entry points form 1 - mu, 1 - lr*weight_decay and lr*sqrt(m/n) on the
 * device with the same operations, so equal values give identical results.
 * Non-finite values in hyper set the non-finite bit of the status word (see
 * dion_get_status); the step still runs.  Argument errors (as for
 * dion_step_batched, plus hyper == NULL or misaligned) return
 * DION_ERR_INVALID_ARG before any launch.
 * This serves a live learning-rate schedule under graph replay (the pages'
 * optimizer takes the learning rate and decay as per-step scalars).
 */
dion_status dion_step_batched_dev(int batch, int m, int n, int r, dion_dtype dt,
                                  void* X, const void* G, float* M, float* Q,
                                  const float* hyper,
                                  void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Upper bound, in bytes, of the fixed device scratch of
 * dion_step_batched_static (64 MiB).  Every GPU that loads libdion holds an
 * array of this size until the process exits.
 */
#define DION_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * dion_step_batched without a workspace argument: the step's scratch memory is
 * a fixed array inside libdion, so the call allocates nothing.  The pages have
 * no counterpart of this entry point; it exists for callers that cannot call
 * cudaMalloc: code whose device memory is all owned by another allocator (a
 * framework's caching pool, or one arena reserved at start-up) and may not
 * take more, and code on a latency-critical path where an allocation, which
 * can synchronize the device, is not acceptable.  The caller still passes
 * X, G, M and Q, with the meaning, layout and in-place updates of
 * dion_step_batched, and the results are those of dion_step_batched.
 *   - Shapes whose dion_workspace_size exceeds DION_STATIC_SCRATCH_BYTES are
 *     rejected with DION_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture, and not from two threads at once.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (the step clears what must start at zero itself).  Calls that
 *     overlap on the GPU (on different streams, or from different threads)
 *     race on it and give wrong results: serialize them.
 *   - The status word is not readable by the caller for this variant: a
 *     rank-deficient P still yields finite output (dependent columns of P
 *     are zeroed) as for dion_step_batched, but a kernel that gave up
 *     waiting (status bit 4 of dion_get_status, outputs undefined) is not
 *     reported either; the call still returns DION_OK.
 */
dion_status dion_step_batched_static(int batch, int m, int n, int r, dion_dtype dt,
                                     void* X, const void* G, float* M, float* Q,
                                     float mu, float lr, float weight_decay, void* cuda_stream);

/*
 * Where this step's panels live inside a dion_step_batched workspace, for
 * callers that want the low-rank factors themselves (diagnostics, or a
 * compressed data-parallel exchange of P and R).  After a step on the
 * caller's stream completes, the workspace holds at byte offset *p_offset the
 * orthonormal P as [batch, m, *p_ld] float32 (first r columns valid), and at
 * *r_offset R = B^T P as [batch, n, *r_ld] float32 (first r columns valid).
 * Same argument rules as dion_workspace_size; any output pointer may be NULL.
 */
dion_status dion_workspace_panels(int batch, int m, int n, int r, dion_dtype dt, size_t* p_offset, int* p_ld,
                                  size_t* r_offset, int* r_ld);

/*
 * Workspace bytes needed by muon_ns_batched for this shape.
 * head_dim = 0 for whole-matrix Newton-Schulz, else n % head_dim must be 0.
 */
dion_status muon_workspace_size(int batch, int m, int n, int head_dim, dion_dtype dt, size_t* bytes);

/*
 * One Muon step on `batch` matrices of shape m x n.
 *   G  [batch, m, n] dt      gradients, read only
 *   M  [batch, m, n] float   momentum (nullable).  If given, M <- mu M + G and
 *                            Newton-Schulz acts on the new M; else on G.
 *   head_dim                 0: orthogonalize each m x n matrix as a whole;
 *                            > 0: orthogonalize each m x head_dim column
 *                            block separately (per-head, n % head_dim == 0).
 *   steps, coeff[3]          `steps` iterations of Y <- a Y + (b A + c A^2) Y,
 *                            A = Y Y^T, after Y <- Y / (||Y||_F + 1e-7); the
 *                            Gram matrix is formed on the smaller side
 *                            (Y is transposed when the block is taller than
 *                            wide).  coeff is a HOST pointer to {a, b, c}.
 *   O  [batch, m, n] dt      orthogonalized update (nullable)
 *   X  [batch, m, n] dt      weights (nullable): X <- (1 - lr*wd) X -
 *                            lr*sqrt(m/n) O, with m, n the matrix's shape
 *                            (also in per-head mode)
 * At least one of X and O must be non-NULL.  dt = DION_BF16 runs the
 * iteration in bfloat16 on the tensor cores with float32 accumulation;
 * dt = DION_F32 runs it in float32.
 */
dion_status muon_ns_batched(int batch, int m, int n, int head_dim, dion_dtype dt,
                            void* X, const void* G, float* M, void* O,
                            int steps, const float* coeff,
                            float mu, float lr, float weight_decay,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Reads the device status word of a workspace used by dion_step_batched or
 * muon_ns_batched (a blocking device-to-host copy of 4 bytes; synchronize
 * the stream of the last call first).  *device_status = 0 means no numeric
 * event; otherwise bits are set:
 *   1  a column of P was found dependent (its part outside the span of the
 *      columns before it is below 1e-6 of its norm): P is rank deficient,
 *      the column was set to zero, the step is valid at the lower rank;
 *   2  a non-finite value was met (input, hyper-parameter or pivot);
 *   4  a pipelined tensor-core kernel gave up waiting on one of its own
 *      internal barriers (after 2 s; a correct run never gets there) and
 *      stopped early: the outputs of that step (X, M, Q) are undefined.
 * The word is cleared at the start of every step.  Returns DION_ERR_NUMERIC
 * when the word is non-zero.
 */
dion_status dion_get_status(const void* workspace, int* device_status);

/* Static, human-readable name of a status code. */
const char* dion_status_string(dion_status s);

/*
 * Per-kernel timing with CUDA events on the launching stream, for
 * measurement.  dion_profile_begin(max_launches) starts recording an event
 * pair around every kernel the library launches (up to max_launches);
 * dion_profile_end() stops.  After the caller has synchronized, entries are
 * read one kernel name at a time: dion_profile_count() names, and
 * dion_profile_entry(i, ...) gives the name (static string), the number of
 * launches and their summed device time in milliseconds.
 * dion_profile_dropped() counts the launches since dion_profile_begin that
 * found all max_launches slots taken and were not timed (the totals then
 * cover only part of the work).  Host-side state is global to the process and
 * not thread-safe.
 */
dion_status dion_profile_begin(int max_launches);
dion_status dion_profile_end(void);
int dion_profile_count(void);
dion_status dion_profile_entry(int i, const char** name, int* launches, double* total_ms);
int dion_profile_dropped(void);

#ifdef __cplusplus
}
#endif

#endif /* DION_H */

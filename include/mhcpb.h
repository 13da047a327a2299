/*
 * mhcpb -- mHC projection/RMS backward for GB300 (sm_103a), C ABI.
 *
 * The operation (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
 * intro):
 *
 *     P  = grad_proj[:, :24]
 *     dX = P @ W + grad_r / (r * K) * X          (stored BF16)
 *     dW = P^T @ X                                (stored FP32)
 *
 * Both matrix products use operands converted to TF32 (round to nearest,
 * ties away) with FP32 accumulation; the RMS term is FP32 arithmetic.  dW is
 * summed over tokens in an order fixed in advance and with no atomic adds, so it is bitwise
 * reproducible for a given (T, K) on any GB300.  Outputs are overwritten,
 * never accumulated into.  grad_proj's columns 24..31 are not read at all.
 *
 * The caller-facing shape of the API follows the same page's "Prepared class
 * API": a plan is created once per shape, reports its scratch size, and each
 * execute launches two kernels on the caller's stream (a streaming kernel
 * that writes dX and per-chunk dW partials into the workspace, then a
 * fixed-order reduction of the partials into dW) and makes no allocation.
 *
 * Layouts (all compact row-major, the page's "Requirements and tensor
 * contract"):
 *     x            BF16 [T, K]
 *     w            FP32 [24, K]
 *     grad_proj    FP32 [T, 32]     columns 24..31 ignored, even NaN/Inf
 *     grad_r, r    FP32 [T]         ([T,1] column vectors); r > 0 required
 *     dx           BF16 [T, K]      output, overwritten
 *     dw           FP32 [24, K]     output, overwritten
 *     grad_x_addend BF16 [T, K]     optional; dX = bf16(fp32(bf16(core)) + fp32(addend)),
 *                                   the value a separate BF16 add would give
 *                                   (prime-kernels PR #15, "fused mHC stream gradient")
 * K counts n_streams * hidden (4 * 5120 = 20480 in the training profile).
 *
 * Ownership: the caller owns every buffer and the stream.  The library keeps
 * no pointer past the return of mhcpb_execute; buffers must stay alive until
 * the enqueued work completes (and for every replay of a captured graph).
 * Executions that may overlap on the GPU need their own workspace and outputs.
 *
 * Errors: every function returns a status.  On any error nothing is enqueued.
 * A wait inside a kernel that runs out of time (about one second) ends the
 * kernel early and records MHCPB_ERR_DEVICE_TIMEOUT in the plan's device
 * status word, read with mhcpb_get_device_status; the outputs of that
 * execution are then undefined but the CUDA context stays usable.
 *
 * Thread safety: a plan may be used from several host threads; executions on
 * one plan share its device status word only.
 */
#ifndef MHCPB_H
#define MHCPB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mhcpb_plan_s* mhcpb_plan_t;

typedef enum {
    MHCPB_OK = 0,
    MHCPB_ERR_INVALID_ARG = 1,        /* NULL plan/pointer, addend presence disagreeing with the plan */
    MHCPB_ERR_UNSUPPORTED_SHAPE = 2,  /* T < 0, K not a positive multiple of 8, or above the maxima below */
    MHCPB_ERR_MISALIGNED = 3,         /* a pointer not 16-byte aligned (4-byte for the gate operands) */
    MHCPB_ERR_ALIASING = 4,           /* two operands (or workspace) share bytes */
    MHCPB_ERR_WRONG_DEVICE = 5,       /* a pointer not in device memory of the plan's device */
    MHCPB_ERR_TF32_NOT_ALLOWED = 6,   /* flags lack MHCPB_ALLOW_TF32 */
    MHCPB_ERR_WORKSPACE_TOO_SMALL = 7,
    MHCPB_ERR_CUDA = 8,               /* a CUDA runtime/driver call failed (see mhcpb_last_cuda_error) */
    MHCPB_ERR_DEVICE_TIMEOUT = 9,     /* reported by mhcpb_get_device_status */
    MHCPB_ERR_UNSUPPORTED_DEVICE = 10, /* device is not compute capability 10.3 (GB300) */
    MHCPB_ERR_SCRATCH_TOO_SMALL = 11  /* mhcpb_execute_static_scratch: the shape needs more
                                         than MHCPB_STATIC_SCRATCH_BYTES of dW partials */
} mhcpb_status_t;

/* Plan flags. */
enum {
    /* Required: the caller accepts TF32 operands in the matrix products (the
     * page makes allow_tf32=True mandatory). */
    MHCPB_ALLOW_TF32 = 1u,
    /* Executions pass a BF16 grad_x_addend that is added into dX. */
    MHCPB_HAS_ADDEND = 2u,
    /* Use the FP32-FMA (CUDA-core) streaming kernel instead of the tensor-core
     * one.  Same results within tolerance, same determinism; kept as the
     * measured control for the tensor-core kernel. */
    MHCPB_FMA_KERNEL = 4u,
    /* Compensated dW reduction: the second kernel sums each element's S chunk
     * partials in the same fixed order, but with an error-free transformation
     * at every addition (TwoSum: s + p = s' + e exactly) and the errors e
     * accumulated beside the sum, then rounds once to FP32: dW = fl(s + E).
     * This is Ogita, Rump and Oishi's cascaded summation (Sum2): as accurate
     * as summing the partials in twice the working precision and rounding
     * once, instead of S - 1 FP32 roundings.  Within a
     * chunk the products are exact in either mode (TF32 x BF16 split into
     * BF16 pairs) and are accumulated by the tensor cores in FP32.  Same
     * determinism: bitwise reproducible and independent of the SM count.
     * The idea comes from the FlashInfer page on
     * cake_rmsnorm_det_train_backward (program windows), whose small-T dw
     * column sums keep exact products, accumulate with TwoSum and round to
     * FP32 once; here it is applied to the cross-chunk reduction.  Costs a
     * few FP32 operations per partial in the second kernel only. */
    MHCPB_COMPENSATED_DW = 8u,
    /* Accumulate dW into the caller's buffer instead of overwriting it:
     * dW_out = dW_in + D in FP32 (one rounding), where D is exactly what the
     * execute would write without this flag (plain or compensated).  For
     * callers that sum weight gradients over micro-batches in an FP32 buffer of
     * their own (prime-kernels PR #15 offers this for its FP8 expert weight
     * gradients; here it applies to dW).  dW must
     * then hold valid values before the execute; dX is unaffected. */
    MHCPB_ACCUMULATE_DW = 16u,
    /* Test hook for failure detection: in the tensor-core kernel the MMA
     * issuer first waits on a barrier that nothing completes, so the execute
     * ends by the in-kernel wait limit, records MHCPB_ERR_DEVICE_TIMEOUT in the
     * status word and leaves the context usable.  Outputs are undefined.  Not
     * for production use. */
    MHCPB_TEST_INJECT_STALL = 1u << 30
};

/* Shape limits (inclusive).  0 <= T <= MHCPB_MAX_T.  T = 0 (an empty batch)
 * is valid everywhere: dX, proj, r and the gate outputs are empty, dW (a sum
 * over no tokens) is written as zeros, or left as dW + 0 with
 * MHCPB_ACCUMULATE_DW, and the workspaces are 0 bytes.  An operand with no
 * elements needs no storage: its pointer may be NULL and is not checked;
 * every non-empty operand (W, dW, the gates' alpha and bias) is checked as
 * for T > 0. */
#define MHCPB_MAX_T (1 << 24)
#define MHCPB_MAX_K (1 << 20)
/* Number of projection columns used, stored width of grad_proj. */
#define MHCPB_NPROJ 24
#define MHCPB_GRAD_PROJ_COLS 32
/* Tokens per dW partial: the token reduction is split into
 * S = ceil(T / MHCPB_PARTIAL_TOKENS(T)) fixed chunks of 512 tokens, whatever
 * the GPU, so dW bits depend only on (T, K) and the inputs. */
#define MHCPB_PARTIAL_TOKENS(T) 512

/* Creates a plan for one shape on one device.  Checks the flags and shape
 * first (no CUDA call is made when they are rejected), then that `device` is
 * a compute-capability-10.3 GPU, loads both kernels and allocates the plan's
 * 4-byte device status word.  `*out` is set only on success. */
mhcpb_status_t mhcpb_plan_create(mhcpb_plan_t* out, int64_t T, int64_t K, int device,
                                 uint32_t flags);

/* Scratch bytes an execute needs: S * 24 * K * 4 with
 * S = ceil(T / MHCPB_PARTIAL_TOKENS(T)) (15,728,640 B at T=4096, K=20480).
 * Contents need no initialisation and are dead after the execute (the
 * reduction drops them from L2 without writing them back when the workspace
 * is 128-byte aligned). */
mhcpb_status_t mhcpb_workspace_bytes(mhcpb_plan_t plan, size_t* bytes);

/* Enqueues the backward on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  All pointers are device pointers on the plan's device,
 * 16-byte aligned and pairwise disjoint; `grad_x_addend` must be NULL unless
 * the plan has MHCPB_HAS_ADDEND, and non-NULL if it has.  Returns without
 * synchronising.  Capturable into a CUDA graph (no allocation, no host sync;
 * tensor maps travel by value in the kernel parameters).  Both kernels are
 * launched as programmatic dependents of the kernel before them in the
 * stream: they may be scheduled early but touch no global memory before it
 * has completed, so stream order holds as for ordinary launches. */
mhcpb_status_t mhcpb_execute(mhcpb_plan_t plan,
                             const void* x, const float* w, const float* grad_proj,
                             const float* grad_r, const float* r,
                             void* dx, float* dw,
                             void* workspace, size_t workspace_bytes,
                             const void* grad_x_addend, void* stream);

/* The same backward in two calls, so that a caller can start using dX (send
 * it, or run the next layer's backward) before dW exists -- the split
 * backward of the prime-kernels PR #15 (the input gradient first, the weight
 * gradients after), applied to this stage:
 *
 *   mhcpb_execute_dx: enqueues the streaming kernel only.  When it completes,
 *   dX is final and `workspace` holds the dW partials of these inputs.
 *   mhcpb_reduce_dw:  enqueues the reduction only: dW from the partials that
 *   the last mhcpb_execute_dx with this workspace left there (overwritten, or
 *   accumulated with MHCPB_ACCUMULATE_DW).  It only reads the workspace, so
 *   it may be repeated on the same partials (e.g. a retried step, or the same
 *   partials accumulated into two dW buffers); each call gives the same sum.
 *   (mhcpb_execute, which writes and reduces the partials in one call, may
 *   drop them from L2 once summed: after it the workspace holds nothing
 *   reusable.)
 *
 * Arguments, checks and status codes are those of mhcpb_execute for the
 * operands each call uses.  The caller orders the two (same stream, or an
 * event) and must not touch the workspace in between.  dX and dW are
 * bitwise identical to mhcpb_execute's. */
mhcpb_status_t mhcpb_execute_dx(mhcpb_plan_t plan,
                                const void* x, const float* w, const float* grad_proj,
                                const float* grad_r, const float* r, void* dx,
                                void* workspace, size_t workspace_bytes,
                                const void* grad_x_addend, void* stream);
mhcpb_status_t mhcpb_reduce_dw(mhcpb_plan_t plan, void* workspace, size_t workspace_bytes,
                               float* dw, void* stream);

/* mhcpb_execute with timing events for measurement tools: records
 * `ev_before` (a cudaEvent_t, may be NULL) before the streaming kernel,
 * `ev_between` after it and `ev_after` after the reduction kernel, all on
 * `stream`.  The recorded event between the kernels stops the reduction from
 * starting early, so use plain mhcpb_execute for end-to-end timing. */
mhcpb_status_t mhcpb_execute_profiled(mhcpb_plan_t plan,
                                      const void* x, const float* w, const float* grad_proj,
                                      const float* grad_r, const float* r,
                                      void* dx, float* dw,
                                      void* workspace, size_t workspace_bytes,
                                      const void* grad_x_addend, void* stream,
                                      void* ev_before, void* ev_between, void* ev_after);

/* Reads (and, if `clear` is nonzero, resets) the plan's device status word.
 * Synchronises with the device.  *status is MHCPB_OK or the first device-side
 * error recorded since the last clear (MHCPB_ERR_DEVICE_TIMEOUT). */
mhcpb_status_t mhcpb_get_device_status(mhcpb_plan_t plan, mhcpb_status_t* status, int clear);

/* Plan facts for tools and tests: which = 0 T, 1 K, 2 partial count S,
 * 3 grid size of the streaming kernel, 4 flags, 5 streaming-kernel dynamic
 * shared memory bytes, 6 token tile, 7 column strip width, 8 tokens per
 * dW partial. */
mhcpb_status_t mhcpb_plan_query(mhcpb_plan_t plan, int which, int64_t* value);

/* Bounds checks of a checked build.  A library compiled with -DMHCPB_CHECKED
 * checks every global-memory access its kernels make at a computed address
 * (tensor-map copies are bounded by their maps) against the extent of its
 * buffer, skips an access found outside and records the first such site of
 * each kernel family.  This call copies those records and clears them:
 * sites[5] = {tensor-core backward, FMA backward, dW reduction, forward, gate
 * kernels}, each 0 (none since the last call) or 1 + the site within that
 * family's source.  *checked is 1 for a checked build; a normal build sets
 * it to 0 and every site to 0 and makes no CUDA call.  NULL arguments:
 * MHCPB_ERR_INVALID_ARG.  The words are per device (the current one) and
 * shared by all plans. */
mhcpb_status_t mhcpb_debug_checked_sites(uint32_t* sites, int* checked);

/* Sets the bound on every wait inside the plan's kernels (default 1 s,
 * accepted range 1 ms .. 60 s).  A wait that runs out ends the kernel early
 * with MHCPB_ERR_DEVICE_TIMEOUT in the status word.  Applies to executes
 * enqueued after the call. */
mhcpb_status_t mhcpb_plan_set_wait_limit(mhcpb_plan_t plan, uint64_t nanoseconds);

/* Caps the persistent grids of the tensor-core backward kernel and of the
 * forward kernel at `max_ctas` CTAs (one per SM; 0 restores the default of
 * every SM), e.g. to leave SMs to kernels that run concurrently on other
 * streams.  Results are bitwise identical for every cap: the dW partition
 * depends only on T, the forward's only on K.  The backward of
 * MHCPB_FMA_KERNEL plans is not affected.  Applies to calls enqueued after
 * this one. */
mhcpb_status_t mhcpb_plan_set_max_ctas(mhcpb_plan_t plan, int max_ctas);

/* Size of the library's built-in scratch buffer (see below): 16 MiB. */
#define MHCPB_STATIC_SCRATCH_BYTES (16u << 20)

/* The backward for callers that cannot allocate device memory at all: code
 * running inside a host framework that owns every byte of the device heap
 * (its own caching allocator, no cudaMalloc allowed), or plugin code that is
 * handed its input and output buffers and nothing else.  Such a caller cannot
 * create a plan (mhcpb_plan_create allocates the plan's status word) nor pass a
 * workspace.  This entry point needs neither: it runs the same two kernels as
 * mhcpb_execute (tensor-core streaming kernel, then the fixed-order reduction)
 * with the dW partials kept in a buffer the library itself declares as a
 * file-scope __device__ array of MHCPB_STATIC_SCRATCH_BYTES.  No counterpart
 * on the pages: their API always takes a caller-allocated workspace.
 *
 *  - No cudaMalloc, cudaFree or other allocating call is made.  The buffer is
 *    part of the loaded module: every GPU that loads the library holds its
 *    16 MiB until the process exits.
 *  - Shapes needing more than that are rejected with
 *    MHCPB_ERR_SCRATCH_TOO_SMALL: S * 24 * K * 4 bytes with
 *    S = ceil(T / MHCPB_PARTIAL_TOKENS(T)), i.e. up to T = 4096 at K = 20480.
 *  - Runs on the calling thread's current device; all pointers must be device
 *    memory there, 16-byte aligned and disjoint (same contract and status codes
 *    as mhcpb_execute).  `flags` must contain MHCPB_ALLOW_TF32 and may contain
 *    MHCPB_HAS_ADDEND (then `grad_x_addend` is required), MHCPB_COMPENSATED_DW
 *    and MHCPB_ACCUMULATE_DW, nothing else.
 *  - The first call on a device does that device's set-up (looks up the
 *    buffer's device address, raises the kernels' shared-memory limit).  Make
 *    that first call before any stream capture.
 *  - Every call, on every stream, shares the one buffer.  Nothing in it needs
 *    to start at zero (each call overwrites every partial it reads) and
 *    nothing in it is meant to be read afterwards (the reduction may drop the
 *    partials from L2 once summed).  Calls that may overlap on the GPU race on
 *    the buffer: order them on one stream or with events.
 *  - Every wait inside the kernels is bounded by a fixed 1 s (there is no plan
 *    to set another limit on).  A wait that runs out leaves the outputs
 *    undefined and is recorded in a device word that the kernels only ever
 *    write: this entry point neither reports nor clears it, so a timeout is
 *    not visible to the caller beyond the wrong outputs. */
mhcpb_status_t mhcpb_execute_static_scratch(int64_t T, int64_t K, uint32_t flags,
                                            const void* x, const float* w, const float* grad_proj,
                                            const float* grad_r, const float* r,
                                            void* dx, float* dw,
                                            const void* grad_x_addend, void* stream);

/* ---------------------------------------------------------------------------
 * The forward of the stage (the step before the backward in the graph).
 * The prime-kernels PR #15 page describes its mhc_projection as the RMS of the
 * streams and the projection logits, both from a single pass over X; this stage's
 * backward (the cuDNN page above) receives the gradients of exactly these two
 * outputs, and its dX formula is their vector-Jacobian product:
 *
 *     proj[t, j] = sum_k X[t, k] * W[j, k]      j < 24, TF32 W (nearest, ties
 *                                                away), FP32 accumulation
 *     r[t]       = sqrt(sum_k X[t, k]^2 / K + eps)
 *
 * Layouts: x BF16 [T, K] and w FP32 [24, K] as for the backward; proj FP32
 * [T, 32] (overwritten; columns 24..31 written as zero, the layout the
 * backward reads grad_proj in); r FP32 [T] (overwritten).  One streaming
 * kernel (tensor cores for the projection, CUDA cores for the squares) and a
 * fixed-order reduction of per-512-column partials: bitwise reproducible and
 * independent of the SM count.  The stream collapse the page's forward also
 * fuses needs weights the pages do not define and is not part of it.
 *
 * Uses the plan's T and K (any flags).  `eps` must be finite and >= 0.
 * Workspace: mhcpb_forward_workspace_bytes (ceil(K/512) * 25 * T' * 4 bytes,
 * T' = T rounded up to 32; 16,384,000 B at T=4096, K=20480), no
 * initialisation needed.  Pointers 16-byte aligned, disjoint, on the plan's
 * device; the same status codes and device status word as mhcpb_execute. */
mhcpb_status_t mhcpb_forward_workspace_bytes(mhcpb_plan_t plan, size_t* bytes);
mhcpb_status_t mhcpb_forward(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                             float* proj, float* r, void* workspace, size_t workspace_bytes,
                             void* stream);
/* mhcpb_forward with timing events for measurement tools (cudaEvent_t, each
 * may be NULL): recorded before the streaming kernel, between the two
 * kernels and after the reduction, on `stream`. */
mhcpb_status_t mhcpb_forward_profiled(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                                      float* proj, float* r, void* workspace,
                                      size_t workspace_bytes, void* stream, void* ev_before,
                                      void* ev_between, void* ev_after);

/* The forward with the gate step fused into its second kernel (the
 * prime-kernels PR #15 page's mhc_projection fuses the gate activations,
 * sigmoid and Sinkhorn, into the projection): writes proj and r exactly as
 * mhcpb_forward does, and h [T, 24] from them exactly as mhcpb_gate_forward
 * (below) would from the stored proj and r with the same alpha, bias and
 * n_iter: the same bits, one kernel launch fewer.  alpha [3], bias [24] and
 * h follow mhcpb_gate_forward's rules (device memory of the plan's device,
 * 4-byte aligned; h overlaps no other operand), the rest mhcpb_forward's.
 * n_iter outside 1 .. MHCPB_GATE_MAX_ITER: MHCPB_ERR_UNSUPPORTED_SHAPE.  The
 * reduction always takes its line layout here. */
mhcpb_status_t mhcpb_forward_gates(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                                   const float* alpha, const float* bias, int n_iter, float* proj,
                                   float* r, float* h, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* ---------------------------------------------------------------------------
 * The gate/normalisation step around the stage: the forward turns the
 * projection logits and r into the mHC gates; the backward turns the gates'
 * upstream gradients into this stage's inputs grad_proj and grad_r.  The
 * cuDNN page (intro) places "the gate and normalization derivatives" before
 * the stage and leaves "Sinkhorn, gate derivatives" to the caller; the
 * prime-kernels PR #15 page ("mhc_projection") fuses "gate activations
 * (sigmoid, Sinkhorn)" into the projection.  Neither page writes the
 * formulas; these calls compute this reading of them (n = 4 streams, so the
 * 24 projection columns are 2n + n^2 logits):
 *
 *     columns 0..3 pre, 4..7 post, 8..23 res (row-major 4 x 4: 8 + 4i + j)
 *     l[t, j]  = a_g(j) * proj[t, j] / r[t] + b[j]       a = (a_pre, a_post, a_res)
 *     H_pre    = sigmoid(l_pre)
 *     H_post   = 2 sigmoid(l_post)
 *     H_res    = Sinkhorn(exp(l_res)): n_iter times, every row divided by its
 *                sum, then every column divided by its sum
 *
 * and the backward, for upstream gradients G in H's layout, the exact chain
 * rule: dl = dL/dl, grad_proj[t, j] = dl[t, j] a_g(j) / r[t] (columns 24..31
 * written as zero), grad_r[t] = -sum_j dl[t, j] a_g(j) proj[t, j] / r[t]^2.
 * The parameter gradients of a and b stay with the caller (the cuDNN page
 * leaves parameter-gradient accumulation to it); `dlogits`, if not NULL,
 * receives dl [T, 24] for that.
 *
 * Layouts (all FP32, row-major): proj [T, 32] (columns 24..31 not read), r [T],
 * alpha [3], bias [24], h and grad_h [T, 24], grad_proj [T, 32], grad_r [T].
 * FP32 arithmetic; results within 1e-4 of each token's largest magnitude of
 * the exact values (the backward for logits spanning up to ~35; beyond ~70 the
 * FP32 backward through the unrolled iterations loses accuracy, though it
 * stays finite; the forward holds at any spread).  0 <= T <= MHCPB_MAX_T, 1 <= n_iter <= MHCPB_GATE_MAX_ITER
 * (else MHCPB_ERR_UNSUPPORTED_SHAPE).  No plan and no workspace: the calls
 * run on the calling thread's current device, where every pointer must be
 * device memory (MHCPB_ERR_WRONG_DEVICE), 4-byte aligned (MHCPB_ERR_MISALIGNED);
 * outputs may not overlap each other or any input (MHCPB_ERR_ALIASING).
 * Enqueued on `stream`; nothing is allocated; outputs are overwritten. */
#define MHCPB_GATE_MAX_ITER 64
mhcpb_status_t mhcpb_gate_forward(int64_t T, int n_iter, const float* proj, const float* r,
                                  const float* alpha, const float* bias, float* h, void* stream);
mhcpb_status_t mhcpb_gate_backward(int64_t T, int n_iter, const float* proj, const float* r,
                                   const float* alpha, const float* bias, const float* grad_h,
                                   float* grad_proj, float* grad_r, float* dlogits, void* stream);

/* Releases the plan (and its status word).  Safe on NULL. */
mhcpb_status_t mhcpb_destroy(mhcpb_plan_t plan);

/* Static description of a status; never NULL. */
const char* mhcpb_status_string(mhcpb_status_t status);

/* The last CUDA error string seen by this thread inside the library (for
 * MHCPB_ERR_CUDA), or "" if none. */
const char* mhcpb_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MHCPB_H */

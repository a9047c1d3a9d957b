/*
 * muonh.h -- C ABI of the B300 (sm_103a) MuonH optimizer-step library.
 *
 * MuonH (Puro-2B digest, jacksunwei.me, section "The load-bearing tricks
 * aren't in the abstract", with its footnote 3 on the Hyperball / MuonH
 * paper): Muon's Newton-Schulz-orthogonalised momentum update, followed by a
 * projection that holds every weight matrix at the Frobenius norm it had at
 * initialisation.  The Puro-2B model card (axforge.ai), section "Training",
 * applies it with zero weight decay to the selected matrix weights and keeps
 * master weights and optimizer state in FP32.
 *
 * One step over a list of matrices W (fp32, rows x cols, row-major), each
 * with gradient G and momentum M (fp32, same shape) and radius r0:
 *
 *   M  <- beta*M + G                               (heavy-ball momentum)
 *   X  <- M / (||M||_F + eps)
 *   ns_steps times, with (a, b, c) = ns_coeffs:
 *       rows <= cols:  A = X X^T;  B = b*A + c*A A;  X <- a*X + B X
 *       rows >  cols:  A = X^T X;  B = b*A + c*A A;  X <- a*X + X B
 *     (the second form is the first applied to X^T and transposed back; A
 *     is always s x s, s = min(rows, cols))
 *   O  <- X
 *   U  <- W - lr*O;   W <- r0 * U / ||U||_F;   W_bf16 <- bf16(W)  (RNE)
 *
 * The pages leave open the momentum form, the Newton-Schulz coefficients and
 * step count, eps, which side of a non-square matrix the iteration works on,
 * and any update scaling; here they are explicit arguments or fixed as above
 * (heavy-ball momentum, the Gram on the short side, update scale 1, no
 * weight decay).
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA device (or managed) addresses on the current
 *    device, 16-byte aligned.  Host pointers are plain host memory, read
 *    before the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is stream-ordered and asynchronous unless stated.
 *  - The caller owns every buffer, including the workspace.  The library
 *    allocates no device memory; it keeps a host-side cache of plans (shape
 *    lists and TMA descriptors) and one status word per device.
 *  - Return codes are MUONH_* below.  On a non-zero return nothing was
 *    launched, except MUONH_ERR_CUDA, which means a launch or a CUDA call
 *    failed; muonh_last_error() then describes it (per host thread).
 *  - Non-finite data is not a return code: kernels record it in the device
 *    status word (MUONH_STATUS_*), read with muonh_get_status().
 */
#ifndef MUONH_H
#define MUONH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
#define MUONH_OK                  0
#define MUONH_ERR_INVALID_ARG     1  /* null/misaligned pointer, bad shape, bad scalar */
#define MUONH_ERR_WORKSPACE       2  /* workspace missing, misaligned or too small */
#define MUONH_ERR_UNSUPPORTED     3  /* flag or shape this build does not handle */
#define MUONH_ERR_CUDA            4  /* a CUDA call or kernel launch failed */

/* ---- device status bits (ORed over all matrices and calls until read) ---- */
#define MUONH_STATUS_NONFINITE_INPUT  0x1u  /* ||M||_F non-finite: W left unchanged */
#define MUONH_STATUS_DEGENERATE_NORM  0x2u  /* ||W - lr*O||_F zero or non-finite: W left unchanged */
#define MUONH_STATUS_KERNEL_TIMEOUT   0x4u  /* a pipeline wait gave up; outputs of that call are invalid */

/* ---- flags ---- */
#define MUONH_FLAG_FP32_CHECK  0x1u  /* Newton-Schulz in fp32 CUDA-core GEMMs (accuracy check mode) */
#define MUONH_FLAG_SYNC_DEBUG  0x4u  /* synchronise and check errors after every kernel */
#define MUONH_FLAG_GEMM_1SM    0x8u  /* Newton-Schulz GEMMs on one SM per 128x256 tile instead of the
                                        default CTA pair per 256x256 tile (same results up to bf16
                                        rounding order; for comparison and small problems) */
#define MUONH_FLAG_ONE_STREAM  0x200u /* enqueue every Newton-Schulz launch on the caller's stream
                                        (default: independent buckets also use up to three
                                        library-owned side streams, forked from and joined back
                                        to the caller's stream with events) */
#define MUONH_FLAG_GEMM_ONE_STEP 0x100u /* CTA-pair GEMMs with one 64-wide K step per pipeline stage
                                        (16 KB TMA boxes) instead of two (32 KB boxes, used when K and
                                        the contiguous extent of MN-major operands are multiples of
                                        64); same results bit for bit */
/* Step variants the pages do not name (muonh_step and muon_step; ignored by
 * muonh_orthogonalize): */
#define MUONH_FLAG_NESTEROV    0x2u  /* Newton-Schulz input G + beta*M_new (Nesterov look-ahead)
                                        instead of M_new; the stored momentum is M_new either way */
#define MUONH_FLAG_SCALE_SHAPE 0x10u /* O <- sqrt(max(1, rows/cols)) * O before the update */
#define MUONH_FLAG_SCALE_RMS   0x20u /* O <- 0.2 * sqrt(max(rows, cols)) * O before the update
                                        (not together with MUONH_FLAG_SCALE_SHAPE) */
#define MUONH_FLAG_GRAD_BF16   0x40u /* each muonh_matrix_t.grad points to bfloat16 values (bit
                                        patterns, same shape, 16-byte aligned) instead of fp32 */

/* One weight matrix and its optimizer state.  All device pointers, fp32
 * row-major rows x cols (row stride = cols elements), 16-byte aligned.
 * w_bf16 may be NULL (no bf16 copy written); it holds bfloat16 bit patterns. */
typedef struct muonh_matrix {
    float*       w;       /* in/out: fp32 master weight                     */
    uint16_t*    w_bf16;  /* out (optional): bf16 copy of the new weight    */
    const float* grad;    /* in: gradient                                   */
    float*       mom;     /* in/out: momentum (caller zeroes it at start)   */
    int64_t      rows;    /* >= 1 */
    int64_t      cols;    /* >= 1 */
} muonh_matrix_t;

/* Largest matrix side handled (rows and cols each <= this). */
#define MUONH_MAX_SIDE 65536

/*
 * r0_dev[i] = ||W_i||_F (fp32; accumulated in fp64) for i < n, read from
 * mats[i].w only.  Call once, at initialisation: the digest's MuonH
 * paragraph fixes each matrix's norm at its initial value.  mats is a host
 * array of n >= 1 entries (grad/mom/w_bf16 are ignored and may be NULL);
 * r0_dev is a device array of n floats.  Needs no workspace.
 */
int muonh_capture_norms(const muonh_matrix_t* mats, int n, float* r0_dev, void* stream);

/*
 * Bytes of device workspace muonh_step needs for this list of shapes and
 * flags, written to *bytes.  Depends only on the shapes, n and flags.
 */
int muonh_workspace_size(const muonh_matrix_t* mats, int n, uint32_t flags, size_t* bytes);

/*
 * One MuonH step over mats[0..n) (host array): momentum, Newton-Schulz,
 * hyperball projection, as in the header comment.  Defined by the Puro-2B
 * digest (jacksunwei.me), section "The load-bearing tricks aren't in the
 * abstract" (MuonH: Muon's update with every weight matrix kept at its
 * initial Frobenius norm by projection onto that hypersphere; footnote 4:
 * the Newton-Schulz iterations), and the Puro-2B model card (axforge.ai),
 * section "Training" (zero weight decay on the MuonH group; FP32 master
 * weights and optimizer state).
 *   r0_dev     device array of n radii (from muonh_capture_norms)
 *   lr         step size eta (the effective, already-multiplied rate)
 *   beta       momentum coefficient
 *   ns_steps   Newton-Schulz iterations, 0..64
 *   ns_coeffs  host array {a, b, c}
 *   eps        added to ||M||_F before dividing, >= 0
 *   flags      MUONH_FLAG_*
 *   workspace  device buffer of >= muonh_workspace_size() bytes, 256-byte
 *              aligned, owned by the caller, not read or written by anything
 *              else while the step runs.  Its contents need no initialising.
 * Matrices must not overlap one another.  A matrix whose momentum turns
 * non-finite, or whose ||W - lr*O||_F is zero or non-finite, keeps its W
 * (its momentum is still updated) and sets a status bit.
 */
int muonh_step(const muonh_matrix_t* mats, int n, const float* r0_dev,
               float lr, float beta, int ns_steps, const float ns_coeffs[3], float eps,
               uint32_t flags, void* workspace, size_t ws_bytes, void* stream);

/*
 * One plain Muon step, the optimizer MuonH is measured against: Puro-2B
 * paper part 6, section 4.3.1 "Cost-Saving Factors" (the matched-ladder
 * comparison of MuonH with Muon), and the digest's footnote 3 ("standard
 * weight decay").  The pages give no formula for it; here it is the same
 * momentum and Newton-Schulz as muonh_step, then
 *     W <- (1 - lr*weight_decay) * W - lr*O,   W_bf16 <- bf16(W)  (RNE)
 * (decoupled weight decay), with no norm constraint (no r0).  Arguments as
 * muonh_step; the workspace is sized by muonh_workspace_size for the same
 * list and flags.  A matrix whose momentum turns non-finite keeps its W and
 * sets MUONH_STATUS_NONFINITE_INPUT.
 */
int muon_step(const muonh_matrix_t* mats, int n, float lr, float beta, float weight_decay,
              int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags,
              void* workspace, size_t ws_bytes, void* stream);

/* One tensor of the AdamW group: fp32, any shape, contiguous, numel
 * elements; every pointer 16-byte aligned. */
typedef struct adamw_param {
    float*       p;           /* in/out: parameter                              */
    uint16_t*    p_bf16;      /* out (optional, NULL = skip): bf16 copy of p    */
    const float* grad;        /* in: gradient                                   */
    float*       exp_avg;     /* in/out: first moment m (zero at the start)     */
    float*       exp_avg_sq;  /* in/out: second moment v (zero at the start)    */
    int64_t      numel;       /* >= 1 */
} adamw_param_t;

/*
 * One AdamW step over params[0..n) (host array), for the parameters outside
 * the MuonH group (Puro-2B model card, section "Training": AdamW, weight
 * decay 0.1).  `step` is the 1-based index of this step (bias correction):
 *   m <- beta1*m + (1 - beta1)*g;   v <- beta2*v + (1 - beta2)*g^2
 *   p <- (1 - lr*weight_decay)*p - lr * m_hat / (sqrt(v_hat) + eps)
 *   with m_hat = m / (1 - beta1^step), v_hat = v / (1 - beta2^step);
 *   p_bf16 <- bf16(p) (RNE)
 * beta1, beta2 in [0, 1); eps >= 0 (eps = 0 with v = 0 gives NaN).  Needs
 * no workspace.  Non-finite gradients propagate into p, m and v (no status
 * bit), as in the textbook method.
 */
int adamw_step(const adamw_param_t* params, int n, int step, float lr, float beta1, float beta2,
               float eps, float weight_decay, void* stream);

/*
 * Workspace bytes for muonh_orthogonalize of one rows x cols matrix.
 */
int muonh_orthogonalize_workspace_size(int64_t rows, int64_t cols, uint32_t flags, size_t* bytes);

/* Element types of muonh_orthogonalize's input and output. */
#define MUONH_DTYPE_F32  0   /* fp32 */
#define MUONH_DTYPE_BF16 1   /* bfloat16 bit patterns (uint16) */

/*
 * Newton-Schulz alone (the "X <- ... ; O <- X" lines of the header comment):
 * the orthogonalisation step of Muon that the Puro-2B digest, section "The
 * load-bearing tricks aren't in the abstract" and its footnote 4, names as
 * Muon's cost.  One rows x cols row-major device matrix `in` (element type
 * in_dtype) is normalised by its Frobenius norm and iterated; the result O
 * is written to `out` (same shape, element type out_dtype; bf16 output is
 * the round-to-nearest-even of the fp32 result).  The model card's
 * "Training" section lets state be bf16 or fp32, whichever each needs,
 * hence both types on either side.  `out` may equal `in` when the types match.
 * A bf16 input is widened exactly to fp32 before the iteration.  Same
 * meaning of ns_steps, ns_coeffs, eps, flags and workspace as muonh_step;
 * the workspace size does not depend on the types.  A dtype other than
 * MUONH_DTYPE_F32 / MUONH_DTYPE_BF16 returns MUONH_ERR_UNSUPPORTED before
 * any launch.  A non-finite ||in||_F sets MUONH_STATUS_NONFINITE_INPUT and
 * `out` is then unspecified.
 */
int muonh_orthogonalize(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows, int64_t cols,
                        int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Newton-Schulz alone, like muonh_orthogonalize, for callers that cannot
 * allocate device memory: code running where cudaMalloc is unavailable or
 * forbidden (inside a custom allocator or memory-pool callback, under a
 * fixed device-memory budget, or in a host process that must not grow its
 * device footprint after start-up).  No counterpart on the pages: it is a
 * packaging of the same computation.
 *
 * Scratch comes from one array of MUONH_STATIC_SCRATCH_BYTES that the
 * library holds in device memory (a file-scope __device__ variable), on
 * every device that loads the library, until the process exits.  Shapes
 * whose muonh_orthogonalize_workspace_size() exceeds it are rejected with
 * MUONH_ERR_WORKSPACE and a message (muonh_last_error); 2048 x 2048,
 * 2048 x 4096 and 1024 x 6144 fit.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it, keyed by
 * the device index, for the life of the process; make that first call
 * before any stream capture.  The kept address belongs to the device's
 * primary context: do not call this entry point after cudaDeviceReset, or
 * from a thread whose current context is one created with the driver API
 * (there the array lives at another address).  The call allocates no device
 * memory and calls no cudaMalloc/cudaFree.  All calls share the one array,
 * so two calls that may overlap on the GPU (different streams, or different
 * host threads on one device) race and corrupt each other's results: order
 * them on one stream.  No scratch byte is read before the same call writes
 * it, so stale contents from an earlier call do not matter.  in_dtype and
 * out_dtype as for muonh_orthogonalize.
 */
#define MUONH_STATIC_SCRATCH_BYTES (96u * 1024u * 1024u)
int muonh_orthogonalize_static(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows,
                               int64_t cols, int ns_steps, const float ns_coeffs[3], float eps, uint32_t flags,
                               void* stream);

/*
 * Data-parallel sharding of the step across ranks (each matrix is an
 * independent unit): owner_out[i] (host array of n ints) = the rank in
 * [0, world_size) that steps matrix i.  Greedy longest-processing-time
 * assignment by the Newton-Schulz cost 3 s^2 l + s^3 (s, l the short and long
 * side): matrices in decreasing cost (ties: lower index first) each go to the
 * least-loaded rank (ties: lower rank).  Deterministic, host only, reads
 * only the shapes of mats.  After their steps, ranks exchange the updated
 * weights (each matrix from its owner).
 */
int muonh_partition(const muonh_matrix_t* mats, int n, int world_size, int* owner_out);

/*
 * Synchronises `stream`, then copies the current device's status word to
 * *status_out (host) and clears it.  Blocking.
 */
int muonh_get_status(uint32_t* status_out, void* stream);

/* Static text for a return code. */
const char* muonh_status_string(int code);

/* Text of the last error on this host thread ("" if none). */
const char* muonh_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
int muonh_version(void);

/* ---- tracing: per-kernel timing (no counterpart on the pages) ----
 * While enabled, every kernel this library launches is bracketed by two CUDA
 * events on the launching stream, and its algorithmic work (floating-point
 * operations of the symmetric-aware Newton-Schulz count, or HBM bytes) is
 * recorded.  Disabled by default; enabling resets the accumulators. */
typedef struct muonh_profile_entry {
    const char* name;   /* kernel kind: "momentum", "ns_gram", ...  (static string) */
    int64_t launches;   /* launches recorded */
    double  ms;         /* event-measured busy time, milliseconds: the length of the union of
                           the launches' intervals (launches on different streams may overlap) */
    double  flops;      /* summed algorithmic floating-point operations */
    double  bytes;      /* summed algorithmic HBM bytes */
} muonh_profile_entry_t;

/* Turn recording on (on != 0, accumulators cleared) or off. */
int muonh_profile_enable(int on);

/* Waits for the recorded events, adds their durations into the per-kind
 * totals, and writes up to max_entries kinds with launches > 0 to out (host
 * array); *n_out = number written.  Blocking.  The kind "ns_busy" covers
 * every Newton-Schulz GEMM launch together: the union of their intervals,
 * the sums of their flops and bytes. */
int muonh_profile_read(muonh_profile_entry_t* out, int max_entries, int* n_out);

/* Number of kernels this library has launched in this process (all devices). */
int64_t muonh_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MUONH_H */

/*
 * okls.h -- C ABI of the GB300 Online KL Shampoo (OKLS) preconditioner step.
 *
 * What the library computes (page "Online KL Shampoo", README of the
 * tilde-research release, section "How it works"): for every matrix gradient
 * G (m x n) of a batch of same-shape parameters W,
 *
 *   S_a <- beta2 S_a + (1-beta2)/n (G P_b)(G P_b)^T + eps I          (m x m)
 *   S_b <- beta2 S_b + (1-beta2)/m (P_a G)^T (P_a G) + eps I          (n x n)
 *   P_a <- S_a^(-1/2),  P_b <- S_b^(-1/2)      (same step; coupled Newton-
 *          Schulz, 10 iterations, 27 binary16 GEMMs, fp32 accumulation)
 *   N   = Nesterov momentum with variance correction
 *   U   = P_a N P_b
 *   W   <- W - lr wd (lr/lr_peak) W - lr c_shape U,
 *          c_shape = sqrt(m/n) / (sqrt(m) + sqrt(n)).
 *
 * With okls_config.method = OKLS_METHOD_SHAMPOO the same kernels run the
 * classic Shampoo step the OKLS page refines (optim-book, "Shampoo" chapter,
 * sections "2 x 3 gradient by hand" and Problem 14):
 *
 *   L <- L + G G^T,  R <- R + G^T G        (plain sums; L_0 = R_0 = eps I)
 *   P_L <- L^(-1/4), P_R <- R^(-1/4)        (two chained Newton-Schulz runs:
 *          the square root of the ridged factor, then its inverse square root)
 *   W   <- W - lr wd (lr/lr_peak) W - lr P_L G P_R.
 *
 * Conventions used by every entry point
 *   - Matrices are row-major and contiguous; a batch is `batch` matrices
 *     back to back (the 3-D (N, m, n) parameter of the README's "Batched
 *     matrices" section).  m = rows = fan-out, n = columns = fan-in.
 *   - Pointers named *_dev are device pointers; they must be 256-byte aligned
 *     (any cudaMalloc / PyTorch CUDA allocation is).  The caller owns every
 *     buffer: the library never allocates device memory in okls_step.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *     okls_step and the state calls are asynchronous on that stream.
 *   - Every function returns an okls_status; on failure a message is kept
 *     per thread and returned by okls_last_error().  No C++ exception ever
 *     crosses this boundary.
 */
#ifndef OKLS_H_
#define OKLS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OKLS_ABI_VERSION 3

typedef enum okls_status {
  OKLS_OK = 0,
  OKLS_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad hyperparameter  */
  OKLS_ERR_UNSUPPORTED = 2,  /* shape/dtype/alignment the kernels can't take */
  OKLS_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed            */
  OKLS_ERR_NONFINITE = 4,    /* device flag: non-finite input or iterate     */
  OKLS_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up           */
  OKLS_ERR_NO_DEVICE = 6     /* no CUDA device / wrong architecture          */
} okls_status;

/* Element types of W and G. */
typedef enum okls_dtype { OKLS_F32 = 0, OKLS_BF16 = 1 } okls_dtype;

/* Preconditioner step computed by okls_step. */
typedef enum okls_method {
  OKLS_METHOD_OKLS = 0,    /* Online KL Shampoo (the default)              */
  OKLS_METHOD_SHAMPOO = 1, /* classic Shampoo: summed factors, -1/4 roots */
  OKLS_METHOD_SOAP = 2,    /* SOAP: Adam in the factors' eigenbasis       */
  OKLS_METHOD_CLEAN = 3    /* Clean: Nystrom low-rank bases, block Adam   */
} okls_method;

/* Which piece of state okls_get_state / okls_set_state move.  In Shampoo
 * mode S_a / S_b hold the sums L / R and P_a / P_b their -1/4 roots; M is
 * unused (left at zero).  In SOAP mode S_a / S_b hold the factor EMAs L / R,
 * P_a / P_b their eigenbases Q_L / Q_R (eigenvectors in columns), M the
 * momentum (original space) and V the second moment (eigenbasis).  In Clean
 * mode (rank r) the sizes differ: P_a / P_b are the bases U_L (batch x m x r)
 * and U_R (batch x n x r, orthonormal columns), S_a / S_b their eigenvalues
 * Lambda_L, Lambda_R (batch x r, decreasing), M / V the Main block's moments
 * (batch x r x r), and parts 6-10 the A and B blocks' first moments and the
 * pooled second moments of blocks A, B and C. */
typedef enum okls_state_part {
  OKLS_STATE_M = 0,   /* momentum,                 batch x m x n, fp32 */
  OKLS_STATE_SA = 1,  /* left factor S_a,          batch x m x m, fp32 */
  OKLS_STATE_SB = 2,  /* right factor S_b,         batch x n x n, fp32 */
  OKLS_STATE_PA = 3,  /* left root P_a = S_a^-1/2, batch x m x m, fp32 */
  OKLS_STATE_PB = 4,  /* right root P_b,           batch x n x n, fp32 */
  OKLS_STATE_V = 5,   /* SOAP only: second moment in the eigenbasis,
                         batch x m x n, fp32 (Clean: batch x r x r) */
  OKLS_STATE_MA = 6,  /* Clean only: M_A, batch x m x r, fp32 */
  OKLS_STATE_MB = 7,  /* Clean only: M_B, batch x r x n, fp32 */
  OKLS_STATE_VA = 8,  /* Clean only: v_A, batch x r, fp32 */
  OKLS_STATE_VB = 9,  /* Clean only: v_B, batch x r, fp32 */
  OKLS_STATE_VC = 10  /* Clean only: v_C, batch, fp32 */
} okls_state_part;

/* Bits of the device status word (okls_query_status). */
#define OKLS_DEV_NONFINITE_INPUT 0x1u  /* G (or the momentum) not finite   */
#define OKLS_DEV_NONFINITE_ITER 0x2u   /* a Newton-Schulz iterate overflowed */
#define OKLS_DEV_NONFINITE_UPDATE 0x4u /* the new W holds a non-finite value */
#define OKLS_DEV_TIMEOUT 0x8u          /* a bounded pipeline wait expired   */

/*
 * Hyperparameters of one same-shape batch.  Defaults (okls_config_default)
 * are those of the README's "Hyperparameters" table: lr 0.09434 (also
 * lr_peak), beta1 0.9684, beta2 0.9482, eps 1e-9, weight_decay 0.0303, and
 * 10 Newton-Schulz iterations with plain binary16 operands and ridge 1e-3.
 *
 *   ns_split_iters  0: every Newton-Schulz GEMM takes plain binary16 operands
 *                   (27 GEMMs, the README's design).  s > 0: iterations
 *                   0..s-1 carry each operand as a (hi, lo) binary16 pair and
 *                   multiply hi*hi + hi*lo + lo*hi (three GEMMs per product),
 *                   for factors whose condition number exceeds ~1e3.
 *   ns_lo           lower end l_0 of the sqrt-eigenvalue interval the
 *                   coefficient schedule is optimised for (default 1e-3:
 *                   eigenvalues down to 1e-6 ||S||_F converge).
 *   ridge           rho >= 0: the root is taken of S + rho ||S||_F I
 *                   (default 1e-3).  Binary16 rounding of Y_0 = S/||S||_F
 *                   perturbs eigenvalues by ~2^-12; without a ridge above
 *                   that floor, rank-deficient factors (every m != n matrix
 *                   at its first step) get negative eigenvalues that the
 *                   cubic drives to overflow.  With ns_split_iters = 3 a
 *                   ridge of 1e-4 suffices.
 *   variance_correction  1: N_t is divided by its standard deviation under
 *                   iid unit-variance gradients; 0: plain Nesterov.
 *   eps_every_update 1: +eps I in every factor update (and S_0 = eps I);
 *                   0: only S_0 = eps I.
 *   root_every      k >= 1 (0 means 1): fresh inverse roots at steps
 *                   t = 1, 1+k, 1+2k, ...; the steps in between still update
 *                   the factors and the momentum but whiten with the roots
 *                   of the last refresh (the practice of recomputing Shampoo
 *                   roots every 20-100 steps; k = 1 is the README's
 *                   zero-staleness method).
 *   method          okls_method.  OKLS_METHOD_SOAP (Clean page, Appendix C,
 *                   Algorithm 4): per step G' = Q_L^T G Q_R, M <- b1 M +
 *                   (1-b1) G, M' = Q_L^T M Q_R, V <- b2 V + (1-b2) G'^2,
 *                   N = Q_L [(M'/(1-b1^t)) / (sqrt(V/(1-b2^t)) + eps)] Q_R^T,
 *                   W <- W - lr wd (lr/lr_peak) W - lr N, L <- b2 L + (1-b2) G G^T,
 *                   R <- b2 R + (1-b2) G^T G, and after steps t with
 *                   t % root_every == 0 Q_L, Q_R <- eigenvectors of L, R
 *                   (decreasing eigenvalues, signs aligned with the previous
 *                   basis); eps is Adam's.  Q = I before the first refresh.
 *                   This build runs SOAP for m, n <= 16384 (fp32
 *                   throughout; the eigensolver is warm-started from the
 *                   previous basis: cyclic Jacobi in one CTA per matrix up
 *                   to 128 x 128, batched fp32 GEMMs past that, with a
 *                   logged-rotation Jacobi for sides up to 544 and a
 *                   blocked Jacobi (128 x 128 pair subproblems, rotations
 *                   applied as fp32-accurate panel products on the tensor
 *                   cores) past 544).  On the
 *                   batched path the workspace holds, per matrix, three
 *                   m x n and one max(mn, m^2, n^2) fp32 buffers, and per
 *                   side d three d x d buffers plus, for d <= 544, one more
 *                   and (d > 128) an eigensolver slice of about 3 d^2
 *                   floats, or, past 544, a blocked-Jacobi slice of about
 *                   4 kp^2 floats (kp = d rounded up to a multiple of 128).
 *                   OKLS_SOAP_LARGE=1 selects the batched path for every
 *                   shape, OKLS_SOAP_BLOCKED=1 the blocked solver for every
 *                   side past 128, and OKLS_EIG_CTAS=c caps the
 *                   logged-rotation solver's CTAs per matrix.  Larger
 *                   shapes return OKLS_ERR_UNSUPPORTED.
 *                   OKLS_METHOD_CLEAN (Clean page, Algorithm 1 with the
 *                   sketch of Eqn. (8) and Appendix A, Algorithm 3): at
 *                   steps t = 1, 1+T, 1+2T, ... (T = root_every) U_L,
 *                   Lambda_L <- rank-`rank` Nystrom approximation of
 *                   b2 U_L Lambda_L U_L^T + (1-b2) G G^T (only the second
 *                   term at t = 1), sketched with rank + oversample columns
 *                   and `power_iters` subspace iterations, likewise U_R from
 *                   G^T G, and the moments move to the new bases (Eqns. (14),
 *                   (15)).  Then, with P_L = I - U_L U_L^T, P_R = I - U_R U_R^T:
 *                   S = U_L^T G U_R, G_A = P_L G U_R, G_B = U_L^T G P_R,
 *                   C = P_L G P_R; M, V (entry-wise on S), M_A, v_A (column
 *                   sums of G_A^2), M_B, v_B (row sums of G_B^2), v_C
 *                   (||C||_F^2) are Adam moments with both bias corrections;
 *                   G~ = U_L N(M, V) U_R^T + N(M_A, v_A) U_R^T + U_L N(M_B, v_B)
 *                   + C / (sqrt(v_C / (1-b2^t)) + eps), N(m, v) = (m/(1-b1^t)) /
 *                   (sqrt(v/(1-b2^t)) + eps); W <- W - lr wd (lr/lr_peak) W
 *                   - lr G~.  The sketch's Gaussian draws are an input (see
 *                   okls_step_noise).  This build runs Clean for m, n <=
 *                   16384 and rank + oversample <= 544, in fp32: one CTA per
 *                   factor up to 128 x 128 with rank + oversample <= 64,
 *                   batched GEMMs past that (the workspace then holds four
 *                   max(m, n) x (rank + oversample) panels and one m x n
 *                   buffer per matrix; OKLS_CLEAN_LARGE=1 selects that path
 *                   for every shape).  Larger shapes return
 *                   OKLS_ERR_UNSUPPORTED.
 *   rank, oversample, power_iters  Clean's r >= 1, p >= 0 (r + p <=
 *                   min(m, n)) and q in [0, 16]; zero for the other methods.
 *                   OKLS_METHOD_SHAMPOO ignores beta1, beta2,
 *                   variance_correction and eps_every_update (the sums add
 *                   G G^T and G^T G with weight 1, eps enters only at reset,
 *                   no momentum, no shape multiplier) and applies `ridge` to
 *                   L and R before the first chain; the second chain takes
 *                   no ridge (its input's condition number is at most
 *                   sqrt((1 + ridge) / ridge)).  The workspace grows by one
 *                   fp32 d x d square root per factor.
 */
typedef struct okls_config {
  int64_t batch;
  int64_t m;
  int64_t n;
  int32_t param_dtype; /* okls_dtype of W */
  int32_t grad_dtype;  /* okls_dtype of G */
  float lr_peak;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  int32_t ns_iters;
  int32_t ns_split_iters;
  float ns_lo;
  float ridge;
  int32_t variance_correction;
  int32_t eps_every_update;
  int32_t root_every;
  int32_t method;      /* an okls_method value; 0 = OKLS */
  int32_t rank;        /* Clean only */
  int32_t oversample;  /* Clean only */
  int32_t power_iters; /* Clean only */
  int32_t reserved[3]; /* must be zero */
} okls_config;

typedef struct okls_handle_s *okls_handle;

/* Library ABI version (OKLS_ABI_VERSION). */
int32_t okls_abi_version(void);

/* Message of the last failed call on this thread ("" if none).  The pointer
 * stays valid until the next failing call on the same thread. */
const char *okls_last_error(void);

/* Fill *cfg with the README defaults for a batch of `batch` m x n matrices. */
okls_status okls_config_default(okls_config *cfg, int64_t batch, int64_t m,
                                int64_t n);

/* Bytes of persistent state (M, S_a, S_b, P_a, P_b, fp32, layout owned by the
 * library) and of workspace the caller must provide to okls_create.  The
 * workspace also persists between steps (binary16 copies of P, scales). */
okls_status okls_state_bytes(const okls_config *cfg, size_t *state_bytes,
                             size_t *workspace_bytes);

/*
 * Bind a handle to caller-owned device memory.  Validates cfg, builds the TMA
 * descriptors on the host and uploads them with one synchronous cudaMemcpy
 * into the head of the workspace; allocates no device memory.  The state is
 * NOT initialised: call okls_reset_state (or okls_set_state for every part).
 * The current CUDA device must be the one that owns the buffers, and it must
 * be an sm_103 GPU (OKLS_ERR_NO_DEVICE otherwise).
 */
okls_status okls_create(const okls_config *cfg, void *state_dev,
                        size_t state_bytes, void *workspace_dev,
                        size_t workspace_bytes, okls_handle *out);

/* M = 0, S_a = eps I, S_b = eps I, P_a = I, P_b = I, step counter t = 0
 * (README: eps is added at factor initialisation; P_0 = I is this library's
 * reading of the first step).  Asynchronous on `stream`. */
okls_status okls_reset_state(okls_handle h, void *stream);

/*
 * One OKLS (or, by cfg.method, classic Shampoo) step over the whole batch,
 * asynchronous on `stream`.
 *   W_dev  batch x m x n, param_dtype, updated in place.
 *   G_dev  batch x m x n, grad_dtype, read only.
 *   lr     current learning rate (finite, >= 0); lr_peak is fixed in cfg.
 * Increments the step counter t on the host.  Device-side failures (non-
 * finite inputs or iterates, an expired wait) are recorded in the device
 * status word and reported by okls_query_status; once the word is non-zero
 * the remaining stages of the step skip their writes, and the W update is
 * skipped whenever an earlier stage flagged (a flag raised by the update
 * itself still lets that step's other tiles land).  Factors with d <= 128
 * run their whole Newton-Schulz chain in one fused launch, one CTA per
 * matrix: there a matrix whose chain overflowed keeps its previous root,
 * while the other matrices of that launch commit their new roots; a root
 * and its scale are always committed together.  Factors of 129 to 1024
 * rows run the chain's 19 GEMM stages as one persistent launch whose tiles
 * wait on per-matrix completion counters in the workspace; it is a
 * cooperative launch (all its CTAs, one per SM, resident at once), and it
 * stops at the first status bit, so after a failure inside it some
 * matrices may already hold their new root (with its scale) and others the
 * previous one.  Larger factors run one launch per stage.  The environment
 * variable OKLS_NS_CHAIN=0, read once per process, selects one launch per
 * stage for every size (the results are bit-identical).
 */
okls_status okls_step(okls_handle h, void *W_dev, const void *G_dev, float lr,
                      void *stream);

/*
 * okls_step with the Gaussian draws of Clean's sketch (Clean page, Appendix A,
 * Algorithm 3: Psi ~ N(0, I)) as an input.
 *   noise_dev  device, fp32, batch x (m + n) x (rank + oversample), 16-byte
 *              aligned, read only: per matrix Psi_L (m rows) then Psi_R
 *              (n rows), row-major.  The first refresh (a state without
 *              bases) takes all rank + oversample columns as the sketch;
 *              later refreshes take the first `oversample` columns of each
 *              row beside the previous basis.  Read only on refresh steps
 *              (t = 1, 1+T, ...), where NULL returns OKLS_ERR_INVALID_ARG;
 *              may be NULL on the others.  The other methods ignore it.
 * okls_step(h, ...) is okls_step_noise(h, ..., NULL, stream).  A refresh
 * whose Cholesky factor breaks down raises OKLS_DEV_NONFINITE_ITER; that step
 * then changes neither W nor the state (the step counter still advances).
 */
okls_status okls_step_noise(okls_handle h, void *W_dev, const void *G_dev,
                            float lr, const float *noise_dev, void *stream);

/* Synchronise `stream`, read the device status word into *dev_status (may be
 * NULL) and clear it.  Returns OKLS_ERR_NONFINITE / OKLS_ERR_TIMEOUT when the
 * corresponding bits were set, OKLS_OK otherwise. */
okls_status okls_query_status(okls_handle h, void *stream,
                              uint32_t *dev_status);

/* Copy one part of the fp32 state to / from a caller device buffer of the
 * part's size (see okls_state_part), asynchronously on `stream`.  Setting
 * OKLS_STATE_PA / PB also refreshes the binary16 copies the GEMMs read. */
okls_status okls_get_state(okls_handle h, int32_t part, void *dst_dev,
                           void *stream);
okls_status okls_set_state(okls_handle h, int32_t part, const void *src_dev,
                           void *stream);

/* Host-side step counter t (the number of completed steps). */
okls_status okls_get_step(okls_handle h, int64_t *t);
okls_status okls_set_step(okls_handle h, int64_t t);

/*
 * Limit of the bounded waits inside the step's tcgen05 GEMM launches, and a
 * test hook for the failure path.  The pages have no counterpart (they
 * describe no failure handling); it serves the OKLS_DEV_TIMEOUT contract of
 * the status word above.
 *   cycles         SM clock cycles a pipeline wait may spin before it raises
 *                  OKLS_DEV_TIMEOUT (0: the default, ~4e9 cycles, ~2 s).
 *   unloaded_tile  -1: none.  >= 0: in every GEMM launch of the following
 *                  steps the producer stops before that linear output tile,
 *                  so its consumers' waits run out with none of that CTA's
 *                  copies or MMAs in flight: the launch raises
 *                  OKLS_DEV_TIMEOUT, every later launch of the step returns
 *                  at once, and okls_query_status reports OKLS_ERR_TIMEOUT.
 *                  W, S and P keep their previous values (the momentum M has
 *                  already advanced when the first GEMM launch fails).
 * Applies to the steps launched after the call, until the next call.
 */
okls_status okls_set_wait_limit(okls_handle h, int64_t cycles,
                                int64_t unloaded_tile);

/* Release the handle (its descriptor table lives in the caller's workspace,
 * so nothing on the device is freed).  The caller must not free state or
 * workspace while work of this handle is still queued.  NULL is accepted. */
okls_status okls_destroy(okls_handle h);

/*
 * Launch accounting of okls_step, for measurement.  Kernel launches are
 * always counted; with timing enabled (okls_profile_enable(h, 1)) every GEMM
 * and bandwidth-kernel launch is bracketed by two CUDA events recorded on the
 * step's stream.  Bandwidth bytes are algorithmic: each element read or
 * written once per launch at its stored width (the per-matrix coefficient
 * kernels are counted in kernel_launches only).
 * okls_profile_read synchronises on those events, returns the sums since the
 * previous read and resets them.  FLOPs are algorithmic: 2 M N K per K
 * segment for dense products, M (M+1) K for the symmetric factor products.
 */
typedef struct okls_profile {
  int64_t kernel_launches; /* all library kernels                         */
  int64_t gemm_launches;   /* tcgen05 GEMM launches among them              */
  double gemm_flops;
  double gemm_ms;          /* summed event time of the timed GEMM launches */
  int64_t timed_launches;
  int64_t ns_launches;     /* the Newton-Schulz subset of the GEMMs         */
  double ns_flops;
  double ns_ms;
  int64_t bw_launches;     /* bandwidth kernels (momentum statistics, pack, */
  double bw_bytes;         /* normalise, sums of squares): algorithmic DRAM */
  double bw_ms;            /* bytes and summed event time                   */
  int64_t bw_timed_launches;
} okls_profile;

okls_status okls_profile_enable(okls_handle h, int32_t timing);
okls_status okls_profile_read(okls_handle h, okls_profile *out);

/*
 * Coefficient schedule the library uses (host computation, no GPU needed):
 * for k < iters, a[k], b[k] of T_k = a_k I + b_k Z_k Y_k, the minimax odd
 * cubic on [l_k, u_k] (l_0 = lo, u_0 = 1), and for k <= iters the exponent
 * zexp[k] = ceil(log2(prod_{j<k} a_j)) of the per-step binary16 scale.
 * Arrays must hold iters (a, b) and iters+1 (zexp) entries.
 */
okls_status okls_ns_schedule(int32_t iters, double lo, double *a, double *b,
                             int32_t *zexp);

/*
 * Debug / test entry: inverse square roots of `count` symmetric d x d fp32
 * matrices S_dev by the library's Newton-Schulz chain (same kernels, schedule
 * and precision mode as okls_step with the given iters / split / lo / ridge).
 *   P_dev     out, count x d x d fp32: S^(-1/2).
 *   root_dev  optional out (NULL to skip), count x d x d fp32: S^(1/2) (one
 *             extra GEMM per iteration-9 factor).
 *   trace_dev optional out (NULL to skip), binary16, (3*iters+1) x count x d
 *             x d: slice 3k, 3k+1, 3k+2 holds the stored iterates Y^_k, Z^_k,
 *             T^_k of iteration k (Z^_0 = I is written as zeros), slice
 *             3*iters holds Z^_iters; row-major, unpadded.  In split mode the
 *             slices hold the high halves.
 *   workspace_dev / workspace_bytes: from okls_inv_root_workspace_bytes.
 * Asynchronous on `stream`; errors of the device status word are reported by
 * the returned status only after an explicit synchronisation, so the call
 * itself synchronises `stream` at the end and reads it.
 */
okls_status okls_inv_root_workspace_bytes(int64_t d, int64_t count,
                                          int32_t iters, int32_t split_iters,
                                          size_t *workspace_bytes);
okls_status okls_inv_root(const float *S_dev, float *P_dev, float *root_dev,
                          uint16_t *trace_dev, int64_t d, int64_t count,
                          int32_t iters, int32_t split_iters, float lo,
                          float ridge, void *workspace_dev,
                          size_t workspace_bytes, void *stream);

/*
 * okls_inv_root without any device allocation.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory
 * when they need a root — allocators that must not re-enter themselves (a
 * root computed from inside an allocation callback), embedders whose device
 * pool is fixed at start-up and must not grow.  It computes the same
 * S^(-1/2) as okls_inv_root (plain or split binary16 chain, same schedule,
 * lo and ridge) but takes its scratch from one static device array inside
 * the library instead of a workspace argument.
 *   S_dev, P_dev  as okls_inv_root (count x d x d fp32, caller-owned).
 *   Capacity      okls_inv_root_noalloc_capacity() bytes (32 MiB), held on
 *                 every GPU that loads the library until the process exits;
 *                 a request whose okls_inv_root_workspace_bytes exceeds it is
 *                 rejected with OKLS_ERR_UNSUPPORTED.  With 10 iterations:
 *                 plain chain d = 1024 up to 2 matrices, d = 512 up to 10,
 *                 d = 256 up to 42; split chain d = 1024 one matrix,
 *                 d = 512 up to 5, d = 256 up to 21; d = 2048 never fits.
 *   First call    on each device looks up the array's device address
 *                 (cudaGetSymbolAddress).
 *   Capture       not usable while `stream` is being captured into a CUDA
 *                 graph: like okls_inv_root it uploads a host-side
 *                 descriptor table and synchronises `stream` to read the
 *                 device status word, and both break a capture.
 *   Sharing       every call on a device uses the same array, which keeps the
 *                 previous call's contents (the call clears what must start
 *                 at zero).  Calls whose work overlaps on the GPU — two
 *                 streams, two host threads — race on the array; serialise
 *                 them.
 * No cudaMalloc, cudaFree or other allocating routine is called.  The call
 * synchronises `stream` before returning, on success and on every error, so
 * no work of it is left queued on the shared array.
 */
size_t okls_inv_root_noalloc_capacity(void);
okls_status okls_inv_root_noalloc(const float *S_dev, float *P_dev, int64_t d,
                                  int64_t count, int32_t iters,
                                  int32_t split_iters, float lo, float ridge,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OKLS_H_ */

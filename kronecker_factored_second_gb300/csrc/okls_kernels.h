// Host-side launchers of the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "okls_internal.h"

namespace okls {

struct NormaliseArgs {
  float* S;         // batch x d x d fp32
  int mirror_only;  // 1: only write S's mirrored lower triangle (steps that keep the roots)
  int upper_only;   // 1: only S's upper triangle is current (factor-product output):
                    //    read it and write the mirrored lower triangle back;
                    // 0: S is a full input, symmetrised as (S + S^T)/2, not written
  int d;
  int64_t ld16, mat16;           // binary16 row pitch (multiple of 8) and matrix stride
  __half *Y, *Ylo;               // Y_0 (and its low half in the split mode)
  __half *T, *Tlo;               // T_0
  __half *Z, *Zlo;               // Z_1 = T_0 2^-z_1
  int split_y, split_t, split_z;
  float a0, b0;
  int z1;
  float ridge;
  const float* scal;
  int scal_ld;
  int slot_cprime, slot_sumsq;
  uint32_t* status;
};

// Fused Newton-Schulz chain of factors with d <= 128 (okls_ns_small.cu).
struct SmallNsFactor {
  float* S;             // count x d x d fp32 factor (its lower triangle is written when upper_only)
  int upper_only;       // 1: only S's upper triangle is current (factor-product output)
  int d, count;
  float* P32;           // count x d x d fp32 output P (want_p)
  __half* Ph;           // binary16 copy of P, row pitch ph_ld, matrix stride ph_mat (want_p)
  int64_t ph_ld, ph_mat;
  float* root32;        // optional count x d x d fp32 square root
  int slot_sumsq, slot_cprime, slot_pscale, slot_rscale;
  int slot_pi;          // written with P^ (P = pi P^): a matrix's binary16 root and its scale change together
};
constexpr int kSmallMaxIters = 32;
struct SmallNsArgs {
  SmallNsFactor f[2];
  int nf;
  float* scal;          // per-matrix scalar table [slot][scal_ld]
  int scal_ld;
  float ridge;
  int iters;
  float a[kSmallMaxIters], b[kSmallMaxIters];
  int z[kSmallMaxIters + 1];
  int want_p;           // 0: the last product forms only the square roots
  uint16_t* trace;      // optional, factor 0 only: (3 iters + 1) x trace_count x d x d binary16
  int64_t trace_count;
  uint32_t* status;
};
cudaError_t launch_ns_small(const SmallNsArgs& A, cudaStream_t st);

// SOAP (okls_soap.cu) for m, n <= 128: one CTA per matrix, fp32.
struct SoapArgs {
  int batch, m, n;
  const void* G;        // batch x m x n, fp32 or bf16 (g_bf16)
  void* W;              // batch x m x n, fp32 or bf16 (w_bf16), updated in place
  int g_bf16, w_bf16;
  float *M, *V, *L, *R; // state: momentum, eigenbasis second moment, factors
  const float *QL, *QR; // eigenbases
  float beta1, beta2, eps, lr, decay;
  float bc1, bc2;       // 1/(1-b1^t), 1/(1-b2^t)
  uint32_t* status;
};
struct SoapRefreshArgs {
  int count;            // matrices per factor side
  const float *S0, *S1; // L (count x d0 x d0) and R (count x d1 x d1)
  float *Q0, *Q1;       // their bases: read as the previous ones, overwritten
  int d0, d1;
  int max_sweeps;
  float tol2;           // stop once off-diagonal^2 <= tol2 * diagonal^2
  uint32_t* status;
};
cudaError_t launch_soap_step(const SoapArgs& A, cudaStream_t st);
cudaError_t launch_soap_refresh(const SoapRefreshArgs& A, cudaStream_t st);
cudaError_t launch_soap_reset(float* M, float* V, float* L, float* R, float* QL, float* QR, int batch, int m, int n,
                              cudaStream_t st);

// Clean (m, n <= 128, r + p <= 64): refresh (Nystrom sketches of both
// factors, then the moments moved to the new bases), the block step, reset.
struct CleanArgs {
  int batch, m, n, r, p, q;
  int warm;                          // the state holds bases from an earlier refresh
  const void* G;                     // batch x m x n, fp32 or bf16 (g_bf16)
  void* W;                           // batch x m x n, fp32 or bf16 (w_bf16), updated in place
  int g_bf16, w_bf16;
  const float* noise;                // batch x (m + n) x (r + p): Psi_L rows, then Psi_R rows
  float *UL, *UR, *lamL, *lamR;      // state: bases (m x r, n x r) and their eigenvalues
  float *ULn, *URn, *lamLn, *lamRn;  // workspace: the refreshed ones
  float *Mm, *Vm;                    // Main block moments, r x r
  float *MA, *MB;                    // A block (m x r) and B block (r x n) first moments
  float *vA, *vB, *vC;               // pooled second moments: r, r, 1
  float beta1, beta2, eps;
  float alr, decay;                  // alpha lr; W <- decay W - alpha lr G~
  float bc1, bc2;                    // 1/(1-b1^t), 1/(1-b2^t)
  int max_sweeps;                    // Jacobi sweeps of the thin SVD
  float tol2;
  uint32_t* status;
};
cudaError_t launch_clean_refresh(const CleanArgs& A, cudaStream_t st);
cudaError_t launch_clean_step(const CleanArgs& A, cudaStream_t st);
cudaError_t launch_clean_reset(const CleanArgs& A, cudaStream_t st);

// Clean for large shapes (m, n <= 16384, r + p <= 544): a batched fp32 GEMM
// and the k x k kernels around it, orchestrated by clean_large_refresh /
// clean_large_step.
struct ClGemm {
  const void* A;      // fp32, or bf16 when a_bf16
  const void* B;      // fp32, or bf16 when b_bf16
  float* C;
  int a_bf16, b_bf16;
  int ta, tb;         // A stored K x M / B stored N x K
  int M, N, K;
  int64_t lda, ldb, ldc;
  int64_t sA, sB, sC; // batch strides (elements)
  int batch;
  float alpha, beta;
  const float* beta_dev;  // per-batch beta when not null
  int a_vec, b_vec;       // set by launch_cl_gemm: 16-byte loads allowed
  const uint32_t* status_guard;  // not null: skip the launch once the status word is set
  uint32_t* status;       // not null: the tensor-core path may run (its bounded waits report here)
};
// fp32 products: on the tensor cores (okls_tc3.cu, three-term bf16 split)
// where t3_gemm_eligible holds, else on the CUDA cores (k_cl_gemm).
cudaError_t launch_cl_gemm(const ClGemm& g, cudaStream_t st);
bool t3_gemm_eligible(const ClGemm& g);
cudaError_t launch_t3_gemm(const ClGemm& g, cudaStream_t st);

// Device buffers of the large Clean path; every array is batch-strided.
struct ClLarge {
  int batch, m, n, r, p, q, k;
  int warm;
  float beta1, beta2, eps, alr, decay, bc1, bc2;
  int max_sweeps;
  float tol2;
  uint32_t* status;
  const void* G;
  void* W;
  int g_bf16, w_bf16;
  const float* noise;                 // batch x (m + n) x k
  // state
  float *UL, *UR, *lamL, *lamR, *M, *V, *MA, *MB, *vA, *vB, *vC;
  // workspace
  float *ULn, *URn, *lamLn, *lamRn;   // refreshed bases
  float *Om, *Y, *X, *T1;             // d x k panels (d = max(m, n))
  float *Gram, *Rinv, *WU, *P, *nu;   // k x k, k x k, k x r, k x r, 1
  float *Mn, *Sm, *MAn, *MBn, *vAn, *vBn;  // transported moments (r x r, r x r, m x r, r x n, r, r)
  float *GU, *UG, *S, *Nm, *Cb;       // step: m x r, r x n, r x r, r x r, m x n
  float *part, *cden;                 // sum-of-squares partials (batch x kClParts), 1
  float* KK;                          // k x k scratch past k = 128: batch x 2 (k + 1)^2
};
constexpr int kClParts = 64;
constexpr int kClMaxK = 544;  // largest r + p of the batched-GEMM path
cudaError_t clean_large_refresh(const ClLarge& L, cudaStream_t st, int* launches);
// Eigenvectors of the batch of symmetric d x d matrices A (d <= 128, one CTA
// per matrix in shared memory), reordered by decreasing eigenvalue into Wout
// (d x d, column c = the eigenvector of rank c), each column's sign chosen so
// that its product with column c of P (d x d: the previous basis seen through
// the current one) is >= 0 (P null: signs as the solver leaves them);
// eigenvalues into lam (may be null).  Past 128: launch_eig_rounds.
cudaError_t launch_cl_eig(const float* A, const float* P, float* Wout, float* lam, int d, int batch, int max_sweeps,
                          float tol2, uint32_t* status, cudaStream_t st);
// Eigenvectors of batches of symmetric k x k matrices, 128 < k <= kClMaxK
// (okls_eig.cu): cyclic Jacobi sweeps on one CTA per matrix, the rotations of
// each sweep logged and applied to V by a wide kernel.  Up to two batches
// (sides) of different k in one set of launches.
struct EigSide {
  const float* A;      // count x k x k; its symmetric part is diagonalised
  const float* P;      // count x k x r, or null: column c's sign makes v . P[:, c] >= 0
  const float* nu;     // count, or null: W = eigenvectors, lam = eigenvalues
  float* W;            // count x k x r: the eigenvectors of the r largest eigenvalues (/ sigma with nu)
  float* lam;          // count x r, or null
  float* scratch;      // count x eig_scratch_floats(k), 16-byte aligned
  int k, r, count;     // count = 0: side unused
  int full;            // set by launch_eig_rounds: A kept as a full matrix in L2
};
struct EigPlan {
  EigSide side[2];
  int max_sweeps;      // >= 1
  float tol2;          // stop once the off-diagonal's squared norm <= tol2 x the diagonal's
  const uint32_t* status;
};
size_t eig_scratch_floats(int k);
cudaError_t launch_eig_rounds(const EigPlan& P, cudaStream_t st, int* launches);
cudaError_t launch_cl_prep(const void* G, int g_bf16, float* out, int64_t mn, int batch, uint32_t* status,
                           cudaStream_t st);
cudaError_t clean_large_step(const ClLarge& L, cudaStream_t st, int* launches);

// Blocked Jacobi for the SOAP refresh of sides past kClMaxK (okls_bjacobi.cu):
// diagonalises the symmetric part of A (= Qh^T F Qh) and writes Qout = Qh W,
// columns by decreasing eigenvalue, each column's sign making its product
// with the same column of Qprev >= 0.  Qout may be Qprev.
struct BjSide {
  const float* A;      // count x d x d
  const float* Qh;     // count x d x d
  const float* Qprev;  // count x d x d
  float* Qout;         // count x d x d
  float* scratch;      // count x bj_scratch_floats(d), 16-byte aligned
  int d, count;        // d > 64
};
size_t bj_scratch_floats(int d);
cudaError_t launch_bjacobi(const BjSide& S, int max_sweeps, float tol2, uint32_t* status, cudaStream_t st,
                           int* launches);

// SOAP past one CTA on the batched GEMM (okls_soap_large.cu): m, n up to
// kSoapLargeMax; a side's eigensolve runs in shared memory up to 128, by
// logged rotations up to kClMaxK and by blocked Jacobi past that.
constexpr int kSoapLargeMax = 16384;
// The eigensolvers' stopping rule for a d x d factor: the off-diagonal's
// squared norm at most this times the diagonal's.  The off-diagonal that fp32
// rotations leave grows like 2^-24 sqrt(d) of the matrix, so the rule keeps
// above that floor.
inline float soap_tol2(int64_t d) { return 1e-12f * (d > 128 ? static_cast<float>(d) / 128.0f : 1.0f); }
struct SoapSideBufs {
  float *Qh, *A;  // batch x d x d each
  float* P;       // batch x d x d: Q^^T Q, or (blocked) the previous basis
  float* Wq;      // batch x d x d (sides up to kClMaxK)
  float* KK;      // eigensolver scratch for 128 < d <= kClMaxK: batch x eig_scratch_floats(d)
  float* BJ;      // blocked Jacobi scratch (blocked sides): batch x bj_scratch_floats(d)
  int blocked;    // the side's refresh runs the blocked solver
};
struct SoapLarge {
  int batch, m, n;
  const void* G;
  void* W;
  int g_bf16, w_bf16;
  float *M, *V, *L, *R, *QL, *QR;       // state
  float beta1, beta2, eps, lr, decay, bc1, bc2;
  int max_sweeps;
  float tol2;
  uint32_t* status;
  float *Gf, *Gp, *Mp;                  // workspace: m x n each
  float* T;                             // max(m n, m^2, n^2)
  SoapSideBufs sideL, sideR;
};
cudaError_t soap_large_step(const SoapLarge& S, int refresh, cudaStream_t st, int* launches);

cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t stream);
cudaError_t launch_chain(const ChainLaunch& C, int num_sms, cudaStream_t stream);

// Reductions are deterministic: kernels write per-block (or per-tile) partials
// into fixed slots and a single thread per matrix sums them in order.
constexpr int kMaxStatParts = 1024;
int momentum_parts(int64_t mn);
int sumsq_parts(int64_t dd);

cudaError_t launch_momentum_stats(const void* G, int g_bf16, const float* M, int batch, int64_t mn,
                                  float b1, float kappa, float* part, int64_t part_ld, uint32_t* status,
                                  cudaStream_t st);
// M may be null (no momentum: N = G); Nh may be null (N^ not needed).
cudaError_t launch_coeffs_pre(int batch, int64_t m, int64_t n, float beta2, int shampoo, float* scal,
                              int scal_ld, const float* part, int64_t part_ld, cudaStream_t st);
cudaError_t launch_pack(const void* G, int g_bf16, float* M, __half* Gh, __half* GhT, __half* Nh,
                        int batch, int m, int n, int64_t ldm, int64_t ldn, float b1, float kappa,
                        const float* scal, int scal_ld, const uint32_t* status, cudaStream_t st);
constexpr int kPostRoots = 1;   // c', P and root output scales of the coming chain
constexpr int kPostCommit = 2;  // root scales pi of the chain that just ran
constexpr int kPostUpdate = 4;  // whitening coefficient
cudaError_t launch_coeffs_post(int batch, float ridge, int zK, int zK1, float* scal, int scal_ld, int mode,
                               const uint32_t* status, const float* part_a, int64_t part_a_ld, int64_t npart_a,
                               const float* part_b, int64_t part_b_ld, int64_t npart_b, cudaStream_t st);
cudaError_t launch_normalise(const NormaliseArgs& A, int batch, cudaStream_t st);
cudaError_t launch_sumsq(const float* S, int batch, int64_t dd, float* part, int64_t part_ld, cudaStream_t st);
cudaError_t launch_requant(const float* P, int batch, int d, __half* Ph, __half* PhT, __half* Pl, __half* PlT,
                           int64_t ld16, int64_t mat16, float* scal, int scal_ld, int slot, cudaStream_t st);
cudaError_t launch_reset_factor(float* S, float* P, __half* Ph, __half* PhT, __half* Pl, __half* PlT, int d,
                                int64_t ld16, int64_t mat16, int batch, float eps, float* scal, int scal_ld,
                                int pi_slot, cudaStream_t st);

}  // namespace okls

// SOAP past one CTA (sm_103a): the one-CTA kernels' method on batched fp32
// GEMMs, for m, n up to 16384.
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching", Appendix C, Algorithm 4 (SOAP), with the KPOP page's section on
// Adam in the Kronecker-factored eigenbasis.  The step's two-sided rotations
// G' = Q_L^T G Q_R, M' = Q_L^T M Q_R, N = Q_L N' Q_R^T and the factor updates
// L <- b2 L + (1-b2) G G^T, R <- b2 R + (1-b2) G^T G are launches of the
// batched GEMM; the moments and the update are element-wise.  The refresh
// (after steps t with t % root_every == 0) warm-starts from the previous
// basis Q as the one-CTA kernel does: Q^ = Q (3 I - Q^T Q)/2, then the
// eigenvectors of Q^^T L Q^ by cyclic Jacobi (in shared memory up to d = 128;
// up to 544 the logged-rotation solver of okls_eig.cu, both sides in one set
// of launches; past that the blocked Jacobi of okls_bjacobi.cu), ordered by
// decreasing eigenvalue and sign-aligned with Q, and Q <- Q^ W.
#include <cuda_bf16.h>

#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

namespace {

__device__ __forceinline__ bool sl_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

// M <- b1 M + (1-b1) G  (G already fp32)
__global__ void k_sl_momentum(float* M, const float* G, int64_t mn, float b1, const uint32_t* status) {
  if (sl_flagged(status)) return;
  const int b = blockIdx.y;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    M[b * mn + e] = fmaf(b1, M[b * mn + e], (1.0f - b1) * G[b * mn + e]);
}

// V <- b2 V + (1-b2) G'^2;  N' = (M' bc1) / (sqrt(V bc2) + eps), in place of M'
__global__ void k_sl_adam(float* V, const float* Gp, float* Mp, int64_t mn, float b2, float bc1, float bc2, float eps,
                          const uint32_t* status) {
  if (sl_flagged(status)) return;
  const int b = blockIdx.y;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t o = b * mn + e;
    const float g = Gp[o];
    const float v = fmaf(b2, V[o], (1.0f - b2) * g * g);
    V[o] = v;
    Mp[o] = (Mp[o] * bc1) / (sqrtf(v * bc2) + eps);
  }
}

template <typename WT>
__device__ __forceinline__ float sl_ld(const WT* p);
template <>
__device__ __forceinline__ float sl_ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float sl_ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void sl_st(float* p, float v) { *p = v; }
__device__ __forceinline__ void sl_st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename WT>
__global__ void k_sl_update(WT* W, const float* N, int64_t mn, float decay, float lr, uint32_t* status) {
  if (sl_flagged(status)) return;
  const int b = blockIdx.y;
  bool bad = false;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t o = b * mn + e;
    const float w = fmaf(-lr, N[o], decay * sl_ld<WT>(W + o));
    bad |= !isfinite(w);
    sl_st(W + o, w);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kStNonfiniteUpdate);
}

// X <- 1.5 I - 0.5 X (the polar step's middle factor), d x d per matrix
__global__ void k_sl_polar(float* X, int d) {
  const int b = blockIdx.y;
  const int64_t dd = static_cast<int64_t>(d) * d;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < dd;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    X[b * dd + e] = (e / d == e % d ? 1.5f : 0.0f) - 0.5f * X[b * dd + e];
}

dim3 sl_grid(int64_t elems, int batch) {
  const int64_t g = (elems + 255) / 256;
  return dim3(static_cast<unsigned>(g < 256 ? (g > 0 ? g : 1) : 256), static_cast<unsigned>(batch));
}

struct SlRun {
  const SoapLarge& S;
  cudaStream_t st;
  int* launches;
  cudaError_t err = cudaSuccess;

  void gemm(const float* A, int ta, int64_t lda, int64_t sA, const float* B, int tb, int64_t ldb, int64_t sB, float* C,
            int64_t ldc, int64_t sC, int M, int N, int K, float alpha = 1.0f, float beta = 0.0f,
            const uint32_t* guard = nullptr) {
    if (err != cudaSuccess) return;
    ClGemm g{};
    g.A = A;
    g.B = B;
    g.C = C;
    g.ta = ta;
    g.tb = tb;
    g.M = M;
    g.N = N;
    g.K = K;
    g.lda = lda;
    g.ldb = ldb;
    g.ldc = ldc;
    g.sA = sA;
    g.sB = sB;
    g.sC = sC;
    g.batch = S.batch;
    g.alpha = alpha;
    g.beta = beta;
    g.status_guard = guard;
    g.status = S.status;
    err = launch_cl_gemm(g, st);
    ++*launches;
  }
  template <class F>
  void launch(F&& f) {
    if (err != cudaSuccess) return;
    f();
    err = cudaGetLastError();
    ++*launches;
  }
};

// One side of the refresh: the factor, the basis and the side's buffers.
struct SlSide {
  const float* F;  // the factor (d x d, state)
  float* Q;        // the basis (d x d, state)
  int d;
  const SoapSideBufs* buf;
};

// Q^ = Q (1.5 I - 0.5 Q^T Q);  A = Q^^T F Q^;  P = Q^^T Q (for the signs; the
// blocked solver takes them from the previous basis directly, which it keeps
// in P: T holds Q^T Q for its polar step).
void sl_refresh_prep(SlRun& R, const SlSide& s) {
  const SoapLarge& S = R.S;
  const SoapSideBufs& B = *s.buf;
  const int d = s.d;
  const int64_t sd = static_cast<int64_t>(d) * d;
  float* QtQ = B.blocked ? S.T : B.P;
  R.gemm(s.Q, 1, d, sd, s.Q, 0, d, sd, QtQ, d, sd, d, d, d);
  R.launch([&] { k_sl_polar<<<sl_grid(sd, S.batch), 256, 0, R.st>>>(QtQ, d); });
  R.gemm(s.Q, 0, d, sd, QtQ, 0, d, sd, B.Qh, d, sd, d, d, d);
  R.gemm(s.F, 0, d, sd, B.Qh, 0, d, sd, S.T, d, sd, d, d, d);
  R.gemm(B.Qh, 1, d, sd, S.T, 0, d, sd, B.A, d, sd, d, d, d);
  if (!B.blocked) R.gemm(B.Qh, 1, d, sd, s.Q, 0, d, sd, B.P, d, sd, d, d, d);
}

// Q <- Q^ W (skipped once the status word is set)
void sl_refresh_finish(SlRun& R, const SlSide& s) {
  const int d = s.d;
  const int64_t sd = static_cast<int64_t>(d) * d;
  R.gemm(s.buf->Qh, 0, d, sd, s.buf->Wq, 0, d, sd, s.Q, d, sd, d, d, d, 1.0f, 0.0f, R.S.status);
}

EigSide eig_side(const SoapLarge& S, const SlSide& s) {
  EigSide e{};
  e.A = s.buf->A;
  e.P = s.buf->P;
  e.W = s.buf->Wq;
  e.scratch = s.buf->KK;
  e.k = s.d;
  e.r = s.d;
  e.count = S.batch;
  return e;
}

// The blocked sides: the sweeps from the polar-corrected previous basis, then
// a refinement -- Q^^T F Q^ formed anew from the basis just found (through
// the polar step again) and up to two more sweeps on it.  The solver tracks
// Q^T F Q through hundreds of rounds of fp32 panel products, whose rounding
// adds up; the refinement's sweeps start from the matrix itself, so what is
// left is one sweep's rounding.
void refine_blocked_passes(SlRun& R, const SlSide& sL, const SlSide& sR) {
  const SoapLarge& S = R.S;
  // both passes order and sign the columns against the previous basis (kept
  // in P: near-equal eigenvalues may rank differently in the two passes)
  for (const SlSide* s : {&sL, &sR}) {
    if (R.err != cudaSuccess || !s->buf->blocked) continue;
    R.err = cudaMemcpyAsync(s->buf->P, s->Q, static_cast<size_t>(S.batch) * s->d * s->d * sizeof(float),
                            cudaMemcpyDeviceToDevice, R.st);
  }
  for (int pass = 0; pass < 2; ++pass) {
    for (const SlSide* s : {&sL, &sR}) {
      if (R.err != cudaSuccess || !s->buf->blocked) continue;
      if (pass == 1) sl_refresh_prep(R, *s);
      BjSide bj{};
      bj.A = s->buf->A;
      bj.Qh = s->buf->Qh;
      bj.Qprev = s->buf->P;
      bj.Qout = s->Q;
      bj.scratch = s->buf->BJ;
      bj.d = s->d;
      bj.count = S.batch;
      R.err = launch_bjacobi(bj, pass == 0 ? S.max_sweeps : 2, soap_tol2(s->d), S.status, R.st, R.launches);
    }
  }
}

// Both sides' bases: where both are in the logged-rotation solver's range
// their eigen-decompositions go out in one set of launches (each is one CTA
// per matrix, so this doubles the SMs at work); a blocked side runs its own
// rounds and writes its basis itself.
void sl_refresh(SlRun& R) {
  const SoapLarge& S = R.S;
  const SlSide sL{S.L, S.QL, S.m, &S.sideL};
  const SlSide sR{S.R, S.QR, S.n, &S.sideR};
  sl_refresh_prep(R, sL);
  sl_refresh_prep(R, sR);
  refine_blocked_passes(R, sL, sR);
  EigPlan plan{};
  plan.max_sweeps = S.max_sweeps;
  plan.tol2 = S.tol2;
  plan.status = S.status;
  int nside = 0;
  for (const SlSide* s : {&sL, &sR}) {
    if (R.err != cudaSuccess) break;
    const SoapSideBufs& B = *s->buf;
    if (B.blocked) {
      continue;  // solved (and refined) above
    } else if (s->d > 128) {
      plan.side[nside++] = eig_side(S, *s);
    } else {
      R.err = launch_cl_eig(B.A, B.P, B.Wq, nullptr, s->d, S.batch, S.max_sweeps, S.tol2, S.status, R.st);
      ++*R.launches;
    }
  }
  if (nside > 0 && R.err == cudaSuccess) R.err = launch_eig_rounds(plan, R.st, R.launches);
  if (!S.sideL.blocked) sl_refresh_finish(R, sL);
  if (!S.sideR.blocked) sl_refresh_finish(R, sR);
}

}  // namespace

cudaError_t soap_large_step(const SoapLarge& S, int refresh, cudaStream_t st, int* launches) {
  SlRun R{S, st, launches};
  const int m = S.m, n = S.n;
  const int64_t mn = static_cast<int64_t>(m) * n, mm = static_cast<int64_t>(m) * m, nn = static_cast<int64_t>(n) * n;
  R.launch([&] { launch_cl_prep(S.G, S.g_bf16, S.Gf, mn, S.batch, S.status, st); });
  // G' = Q_L^T (G Q_R)
  R.gemm(S.Gf, 0, n, mn, S.QR, 0, n, nn, S.T, n, mn, m, n, n);
  R.gemm(S.QL, 1, m, mm, S.T, 0, n, mn, S.Gp, n, mn, m, n, m);
  // M <- b1 M + (1-b1) G;  M' = Q_L^T (M Q_R)
  R.launch([&] { k_sl_momentum<<<sl_grid(mn, S.batch), 256, 0, st>>>(S.M, S.Gf, mn, S.beta1, S.status); });
  R.gemm(S.M, 0, n, mn, S.QR, 0, n, nn, S.T, n, mn, m, n, n);
  R.gemm(S.QL, 1, m, mm, S.T, 0, n, mn, S.Mp, n, mn, m, n, m);
  // V and N' (in place of M')
  R.launch([&] {
    k_sl_adam<<<sl_grid(mn, S.batch), 256, 0, st>>>(S.V, S.Gp, S.Mp, mn, S.beta2, S.bc1, S.bc2, S.eps, S.status);
  });
  // N = (Q_L N') Q_R^T, into G' (no longer needed)
  R.gemm(S.QL, 0, m, mm, S.Mp, 0, n, mn, S.T, n, mn, m, n, m);
  R.gemm(S.T, 0, n, mn, S.QR, 1, n, nn, S.Gp, n, mn, m, n, n);
  R.launch([&] {
    if (S.w_bf16)
      k_sl_update<__nv_bfloat16><<<sl_grid(mn, S.batch), 256, 0, st>>>(static_cast<__nv_bfloat16*>(S.W), S.Gp, mn,
                                                                        S.decay, S.lr, S.status);
    else
      k_sl_update<float><<<sl_grid(mn, S.batch), 256, 0, st>>>(static_cast<float*>(S.W), S.Gp, mn, S.decay, S.lr,
                                                                S.status);
  });
  // L <- b2 L + (1-b2) G G^T;  R <- b2 R + (1-b2) G^T G
  R.gemm(S.Gf, 0, n, mn, S.Gf, 1, n, mn, S.L, m, mm, m, m, n, 1.0f - S.beta2, S.beta2, S.status);
  R.gemm(S.Gf, 1, n, mn, S.Gf, 0, n, mn, S.R, n, nn, n, n, m, 1.0f - S.beta2, S.beta2, S.status);
  if (refresh) sl_refresh(R);
  return R.err;
}

}  // namespace okls

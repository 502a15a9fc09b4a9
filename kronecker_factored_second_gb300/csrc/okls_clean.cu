// Clean (Nystrom low-rank factors with block-wise Adam) for m, n <= 128 and
// r + p <= 64 (sm_103a).
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching": Algorithm 1 (the step), Eqn. (8) (the sketch A Omega of
// b2 U Lambda U^T + (1-b2) G G^T without forming it), Appendix A Algorithm 3
// (warm-started Nystrom with subspace iteration), Eqns. (10)-(13) and
// Table 1 (blocks Main, A, B, C and their moments), Eqns. (14)-(15) (moments
// moved to refreshed bases) and Eqn. (16) (the update).
//
// One CTA per (matrix, side) for the refresh and one per matrix for the
// moment transport and the step; fp32 in shared memory on the CUDA cores,
// every product on staged operands with 4 x 4 register tiles (at these
// sizes a product is at most ~1 M FMAs and the bases must be fp32-accurate,
// so neither the tensor cores nor binary16 operands are used).
// The thin QRs are classical Gram-Schmidt applied twice (robust on the
// ill-conditioned power-iterated sketch), the k x k Cholesky is right-looking,
// the thin SVD of Y_nu C^-1 comes from a cyclic Jacobi eigensolve of its
// Gram matrix, and nu is the binary32 spacing at the spectral norm of Y (the
// working precision's eps).
#include <cuda_bf16.h>

#include "okls_internal.h"
#include "okls_kernels.h"
#include "okls_tile.cuh"

namespace okls {

constexpr int kCMax = 128;   // m, n
constexpr int kCK = 64;      // r + p
constexpr int kCThreads = 256;
// Staged-operand pitches: odd, so that the rows a warp's 4 x 4 tiles read at
// one k fall into distinct banks.
constexpr int kPG = kCMax + 1;  // m x n and r x n operands
constexpr int kPU = kCK + 1;    // m x r, n x r and r x r operands

// ------------------------------------------------------------- block helpers
__device__ __forceinline__ float c_block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
  return s;  // every thread
}

// Orthonormalise the k columns of X (d x k, pitch ld) in place: classical
// Gram-Schmidt twice per column; R's diagonal comes out non-negative.
__device__ void c_qr(float* X, int ld, int d, int k, float* coef, float* red) {
  for (int j = 0; j < k; ++j) {
    for (int pass = 0; pass < 2; ++pass) {
      // coef[i] = <x_i, x_j>, i < j
      for (int i = threadIdx.x >> 5; i < j; i += blockDim.x >> 5) {
        float s = 0.0f;
        for (int row = threadIdx.x & 31; row < d; row += 32) s = fmaf(X[row * ld + i], X[row * ld + j], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((threadIdx.x & 31) == 0) coef[i] = s;
      }
      __syncthreads();
      for (int row = threadIdx.x; row < d; row += blockDim.x) {
        float v = X[row * ld + j];
        for (int i = 0; i < j; ++i) v = fmaf(-coef[i], X[row * ld + i], v);
        X[row * ld + j] = v;
      }
      __syncthreads();
    }
    float s = 0.0f;
    for (int row = threadIdx.x; row < d; row += blockDim.x) s = fmaf(X[row * ld + j], X[row * ld + j], s);
    const float nrm = sqrtf(c_block_sum(s, red));
    const float inv = nrm > 0.0f ? 1.0f / nrm : 0.0f;
    for (int row = threadIdx.x; row < d; row += blockDim.x) X[row * ld + j] *= inv;
    __syncthreads();
  }
}

// Eigen-decomposition of the symmetric k x k matrix A (pitch kPU) by
// cyclic Jacobi: A ends diagonal, V holds the eigenvectors in columns.
__device__ void c_jacobi(float* A, float* V, int k, float* cs, int* pr, float* red, int max_sweeps, float tol2) {
  const int dp = k + (k & 1), np = dp / 2;
  for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
    const int i = e / dp, j = e % dp;
    if (i >= k || j >= k) A[i * kPU + j] = 0.0f;
    V[i * kPU + j] = i == j ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    float off = 0.0f, dg = 0.0f;
    for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
      const int i = e / dp, j = e % dp;
      const float v = A[i * kPU + j];
      if (i == j)
        dg = fmaf(v, v, dg);
      else
        off = fmaf(v, v, off);
    }
    const float offs = c_block_sum(off, red);
    const float dgs = c_block_sum(dg, red);
    if (!(offs > tol2 * dgs)) break;
    for (int rd = 0; rd < dp - 1; ++rd) {
      for (int q = threadIdx.x; q < np; q += blockDim.x) {
        auto idx = [&](int pos) { return pos == 0 ? 0 : 1 + (pos - 1 + rd) % (dp - 1); };
        int p = idx(q), r = idx(dp - 1 - q);
        if (p > r) {
          const int x = p;
          p = r;
          r = x;
        }
        const float apq = A[p * kPU + r];
        float c = 1.0f, s = 0.0f;
        if (apq != 0.0f) {
          const float th = (A[r * kPU + r] - A[p * kPU + p]) / (2.0f * apq);
          const float t = copysignf(1.0f, th) / (fabsf(th) + sqrtf(fmaf(th, th, 1.0f)));
          c = rsqrtf(fmaf(t, t, 1.0f));
          s = t * c;
        }
        cs[2 * q] = c;
        cs[2 * q + 1] = s;
        pr[2 * q] = p;
        pr[2 * q + 1] = r;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * dp; e += blockDim.x) {
        const int q = e / dp, j = e % dp;
        const int p = pr[2 * q], r = pr[2 * q + 1];
        const float c = cs[2 * q], s = cs[2 * q + 1];
        const float ap = A[p * kPU + j], ar = A[r * kPU + j];
        A[p * kPU + j] = c * ap - s * ar;
        A[r * kPU + j] = s * ap + c * ar;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * dp; e += blockDim.x) {
        const int q = e / dp, i = e % dp;
        const int p = pr[2 * q], r = pr[2 * q + 1];
        const float c = cs[2 * q], s = cs[2 * q + 1];
        const float ap = A[i * kPU + p], ar = A[i * kPU + r];
        A[i * kPU + p] = c * ap - s * ar;
        A[i * kPU + r] = s * ap + c * ar;
        const float vp = V[i * kPU + p], vr = V[i * kPU + r];
        V[i * kPU + p] = c * vp - s * vr;
        V[i * kPU + r] = s * vp + c * vr;
      }
      __syncthreads();
    }
  }
}

// An earlier stage flagged the status word: one read per block, so that every
// thread of the block takes the same branch.
__device__ __forceinline__ bool c_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

// spacing of binary32 numbers at x > 0
__device__ __forceinline__ float c_eps32(float x) { return x > 0.0f ? ldexpf(1.0f, ilogbf(x) - 23) : 0.0f; }

template <typename GT>
__device__ __forceinline__ float c_gload(const GT* p);
template <>
__device__ __forceinline__ float c_gload<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float c_gload<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// ------------------------------------------------------------------ refresh
// Shared-memory plan of the refresh (floats).  The k x k region holds the
// previous basis while the sketch is applied, then Omega^T Y_nu (Cholesky),
// Z^T Z (Jacobi) and the eigenvectors.
constexpr int kRG = 0;                          // G                    (m x n, pitch kPG)
constexpr int kROm = kRG + kCMax * kPG;         // Omega                (d x k, pitch kPU)
constexpr int kRY = kROm + kCMax * kPU;         // Y, Y_nu, Z           (d x k)
constexpr int kRT = kRY + kCMax * kPU;          // G^T X / G X / U^T X; the new basis (d x k)
constexpr int kRK = kRT + kCMax * kPU;          // U_prev (d x r), then K1, K2, K3 (k x k each)
constexpr int kRVec = kRK + 3 * kCK * kPU;      // 4 kCK floats, 2 kCK floats, 2 kCK ints
constexpr int kRefreshFloats = kRVec + 8 * kCK;

// Block (matrix b, side s): s = 0 sketches L (d = m), s = 1 sketches R (d = n).
template <typename GT>
__global__ void __launch_bounds__(kCThreads) k_clean_refresh(CleanArgs A) {
  extern __shared__ float sm[];
  if (c_flagged(A.status)) return;
  const int side = blockIdx.x < A.batch ? 0 : 1;
  const int b = side == 0 ? blockIdx.x : blockIdx.x - A.batch;
  const int m = A.m, n = A.n, r = A.r, k = A.r + A.p;
  const int d = side == 0 ? m : n, o = side == 0 ? n : m;  // sketched and other dimension
  float* Gs = sm + kRG;
  float* Om = sm + kROm;
  float* Yb = sm + kRY;
  float* Tb = sm + kRT;
  float* Us = sm + kRK;                  // U_prev while the sketch is applied
  float* K1 = sm + kRK;
  float* K2 = K1 + kCK * kPU;
  float* K3 = K2 + kCK * kPU;
  float* vec = sm + kRVec;               // 4 * kCK
  float* cs = vec + 4 * kCK;             // 2 * kCK
  int* pr = reinterpret_cast<int*>(cs + 2 * kCK);  // 2 * kCK
  __shared__ float red[kCThreads / 32];
  __shared__ float scal[2];
  const GT* G = static_cast<const GT*>(A.G) + static_cast<int64_t>(b) * m * n;
  const float* Uold = (side == 0 ? A.UL : A.UR) + static_cast<int64_t>(b) * d * r;
  const float* lold = (side == 0 ? A.lamL : A.lamR) + static_cast<int64_t>(b) * r;
  float* Unew = (side == 0 ? A.ULn : A.URn) + static_cast<int64_t>(b) * d * r;
  float* lnew = (side == 0 ? A.lamLn : A.lamRn) + static_cast<int64_t>(b) * r;
  const float* noise = A.noise + static_cast<int64_t>(b) * (m + n) * k + (side == 0 ? 0 : static_cast<int64_t>(m) * k);

  for (int e = threadIdx.x; e < m * n; e += blockDim.x) Gs[(e / n) * kPG + e % n] = c_gload<GT>(G + e);
  // Omega = [U_prev, Psi] (warm) or Psi (cold), then orthonormalised (reading c1)
  for (int e = threadIdx.x; e < d * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    float v;
    if (A.warm)
      v = j < r ? Uold[i * r + j] : noise[i * k + (j - r)];
    else
      v = noise[i * k + j];
    Om[i * kPU + j] = v;
  }
  if (A.warm)
    for (int e = threadIdx.x; e < d * r; e += blockDim.x) Us[(e / r) * kPU + e % r] = Uold[e];
  __syncthreads();
  c_qr(Om, kPU, d, k, vec, red);
  // Y = A X with A = b2 U Lambda U^T + (1-b2) G G^T (L side) or G^T G (R side)
  const float w2 = 1.0f - A.beta2;
  auto apply = [&](const float* X, float* Y) {
    if (side == 0) {
      tile_mm4(Gs, kPG, true, X, kPU, false, o, k, d, [&](int i, int j, float v) { Tb[i * kPU + j] = v; });
      __syncthreads();
      tile_mm4(Gs, kPG, false, Tb, kPU, false, d, k, o, [&](int i, int j, float v) { Y[i * kPU + j] = w2 * v; });
    } else {
      tile_mm4(Gs, kPG, false, X, kPU, false, o, k, d, [&](int i, int j, float v) { Tb[i * kPU + j] = v; });
      __syncthreads();
      tile_mm4(Gs, kPG, true, Tb, kPU, false, d, k, o, [&](int i, int j, float v) { Y[i * kPU + j] = w2 * v; });
    }
    __syncthreads();
    if (A.warm) {
      // + b2 U (Lambda (U^T X))
      tile_mm4(Us, kPU, true, X, kPU, false, r, k, d, [&](int i, int j, float v) { Tb[i * kPU + j] = lold[i] * v; });
      __syncthreads();
      tile_mm4(Us, kPU, false, Tb, kPU, false, d, k, r,
            [&](int i, int j, float v) { Y[i * kPU + j] = fmaf(A.beta2, v, Y[i * kPU + j]); });
      __syncthreads();
    }
  };
  for (int it = 0; it < A.q; ++it) {
    apply(Om, Yb);
    for (int e = threadIdx.x; e < d * k; e += blockDim.x) Om[(e / k) * kPU + e % k] = Yb[(e / k) * kPU + e % k];
    __syncthreads();
    c_qr(Om, kPU, d, k, vec, red);
  }
  apply(Om, Yb);
  // nu = eps(||Y||_2): ||Y||_2^2 = largest eigenvalue of Y^T Y, by 60 power
  // steps in one warp (k <= 64: two entries per lane, no block barriers)
  tile_mm4(Yb, kPU, true, Yb, kPU, false, k, k, d, [&](int i, int j, float v) { K1[i * kPU + j] = v; });
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int j = lane; j < k; j += 32) vec[j] = 1.0f;
    __syncwarp();
    float nrm = 0.0f;
    for (int it = 0; it < 60; ++it) {
      float s2 = 0.0f;
      for (int i = lane; i < k; i += 32) {
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s = fmaf(K1[i * kPU + j], vec[j], s);
        vec[kCK + i] = s;
        s2 = fmaf(s, s, s2);
      }
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o2);
      nrm = sqrtf(s2);  // -> lambda_max of Y^T Y
      __syncwarp();
      for (int i = lane; i < k; i += 32) vec[i] = nrm > 0.0f ? vec[kCK + i] / nrm : 0.0f;
      __syncwarp();
    }
    if (lane == 0) scal[0] = nrm;
  }
  __syncthreads();
  const float nu = c_eps32(sqrtf(scal[0]));
  // Y_nu = Y + nu Omega;  B = Omega^T Y_nu;  C = chol((B + B^T)/2), upper
  for (int e = threadIdx.x; e < d * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    Yb[i * kPU + j] = fmaf(nu, Om[i * kPU + j], Yb[i * kPU + j]);
  }
  __syncthreads();
  tile_mm4(Om, kPU, true, Yb, kPU, false, k, k, d, [&](int i, int j, float v) { K1[i * kPU + j] = v; });
  __syncthreads();
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    K2[i * kPU + j] = 0.5f * (K1[i * kPU + j] + K1[j * kPU + i]);
  }
  __syncthreads();
  // right-looking Cholesky of K2 into its lower triangle: K2 = Lc Lc^T, C = Lc^T
  bool bad = false;
  for (int j = 0; j < k; ++j) {
    if (threadIdx.x == 0) {
      const float djj = K2[j * kPU + j];
      scal[1] = djj > 0.0f ? sqrtf(djj) : 0.0f;
    }
    __syncthreads();
    const float cj = scal[1];
    if (!(cj > 0.0f)) bad = true;
    for (int i = j + threadIdx.x; i < k; i += blockDim.x)
      K2[i * kPU + j] = i == j ? cj : (cj > 0.0f ? K2[i * kPU + j] / cj : 0.0f);
    __syncthreads();
    for (int e = threadIdx.x; e < (k - j - 1) * (k - j - 1); e += blockDim.x) {
      const int i = j + 1 + e / (k - j - 1), l = j + 1 + e % (k - j - 1);
      if (l <= i) K2[i * kPU + l] = fmaf(-K2[i * kPU + j], K2[l * kPU + j], K2[i * kPU + l]);
    }
    __syncthreads();
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) atomicOr(A.status, kStNonfiniteIter);
    return;
  }
  // Z = Y_nu C^-1 = Y_nu Lc^-T: row by row, z Lc^T = y (forward substitution)
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    for (int j = 0; j < k; ++j) {
      float v = Yb[i * kPU + j];
      for (int l = 0; l < j; ++l) v = fmaf(-Yb[i * kPU + l], K2[j * kPU + l], v);
      Yb[i * kPU + j] = v / K2[j * kPU + j];
    }
  }
  __syncthreads();
  // thin SVD of Z: eigen-decomposition of Z^T Z = V Sigma^2 V^T
  tile_mm4(Yb, kPU, true, Yb, kPU, false, k, k, d, [&](int i, int j, float v) { K1[i * kPU + j] = v; });
  __syncthreads();
  c_jacobi(K1, K3, k, cs, pr, red, A.max_sweeps, A.tol2);
  // order by decreasing Sigma^2: rank of each eigenvalue
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const float lj = K1[j * kPU + j];
    int rank = 0;
    for (int i = 0; i < k; ++i) {
      const float li = K1[i * kPU + i];
      rank += (li > lj) || (li == lj && i < j);
    }
    pr[j] = rank;
    vec[2 * kCK + rank] = lj;
  }
  __syncthreads();
  // U[:, rank] = Z v_j / sigma_j for the r leading ranks; Lambda = max(0, Sigma^2 - nu)
  tile_mm4(Yb, kPU, false, K3, kPU, false, d, k, k, [&](int i, int j, float v) {
    const int rank = pr[j];
    if (rank < r) {
      const float s2 = K1[j * kPU + j];
      Tb[i * kPU + rank] = s2 > 0.0f ? v * rsqrtf(s2) : 0.0f;
    }
  });
  __syncthreads();
  // sign alignment with the previous basis (warm start)
  for (int j = threadIdx.x; j < r; j += blockDim.x) {
    float s = 1.0f;
    if (A.warm) {
      float dot = 0.0f;
      for (int i = 0; i < d; ++i) dot = fmaf(Tb[i * kPU + j], Uold[i * r + j], dot);
      s = dot < 0.0f ? -1.0f : 1.0f;
    }
    cs[j] = s;
    lnew[j] = fmaxf(0.0f, vec[2 * kCK + j] - nu);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < d * r; e += blockDim.x) {
    const int i = e / r, j = e % r;
    Unew[e] = cs[j] * Tb[i * kPU + j];
  }
}

// ------------------------------------------------------------ moment transport
// Eqns. (14)-(15) with O_L = U_L,new^T U_L,old and O_R = U_R,old^T U_R,new;
// then the new bases become the current ones.  Shared-memory plan (floats):
constexpr int kXBuf = kCMax * kPU;             // >= m x r (pitch kPU) and r x n (pitch kPG)
constexpr int kXULn = 0;                       // U_L,new       (m x r, pitch kPU)
constexpr int kXURn = kXULn + kXBuf;           // U_R,new       (n x r)
constexpr int kXS1 = kXURn + kXBuf;            // scratch
constexpr int kXS2 = kXS1 + kXBuf;             // scratch
constexpr int kXOL = kXS2 + kXBuf;             // O_L           (r x r, pitch kPU)
constexpr int kXOR = kXOL + kCK * kPU;         // O_R
constexpr int kRotateFloats = kXOR + kCK * kPU;

__global__ void __launch_bounds__(kCThreads) k_clean_rotate(CleanArgs A) {
  extern __shared__ float sm[];
  if (c_flagged(A.status)) return;
  const int b = blockIdx.x;
  const int m = A.m, n = A.n, r = A.r;
  float* UL = A.UL + static_cast<int64_t>(b) * m * r;
  float* UR = A.UR + static_cast<int64_t>(b) * n * r;
  const float* ULn = A.ULn + static_cast<int64_t>(b) * m * r;
  const float* URn = A.URn + static_cast<int64_t>(b) * n * r;
  if (A.warm) {
    float* M = A.Mm + static_cast<int64_t>(b) * r * r;
    float* MA = A.MA + static_cast<int64_t>(b) * m * r;
    float* MB = A.MB + static_cast<int64_t>(b) * r * n;
    float* vA = A.vA + static_cast<int64_t>(b) * r;
    float* vB = A.vB + static_cast<int64_t>(b) * r;
    float* Ln = sm + kXULn;
    float* Rn = sm + kXURn;
    float* S1 = sm + kXS1;
    float* S2 = sm + kXS2;
    float* OL = sm + kXOL;
    float* OR = sm + kXOR;
    for (int e = threadIdx.x; e < m * r; e += blockDim.x) {
      Ln[(e / r) * kPU + e % r] = ULn[e];
      S1[(e / r) * kPU + e % r] = UL[e];
    }
    for (int e = threadIdx.x; e < n * r; e += blockDim.x) {
      Rn[(e / r) * kPU + e % r] = URn[e];
      S2[(e / r) * kPU + e % r] = UR[e];
    }
    __syncthreads();
    tile_mm4(Ln, kPU, true, S1, kPU, false, r, r, m, [&](int i, int j, float v) { OL[i * kPU + j] = v; });
    tile_mm4(S2, kPU, true, Rn, kPU, false, r, r, n, [&](int i, int j, float v) { OR[i * kPU + j] = v; });
    __syncthreads();
    // M <- O_L M O_R
    for (int e = threadIdx.x; e < r * r; e += blockDim.x) S1[(e / r) * kPU + e % r] = M[e];
    __syncthreads();
    tile_mm4(OL, kPU, false, S1, kPU, false, r, r, r, [&](int i, int j, float v) { S2[i * kPU + j] = v; });
    __syncthreads();
    tile_mm4(S2, kPU, false, OR, kPU, false, r, r, r, [&](int i, int j, float v) { M[i * r + j] = v; });
    __syncthreads();
    // M_A <- (I - U_Ln U_Ln^T) M_A O_R:  T = M_A O_R, X = U_Ln^T T, M_A = T - U_Ln X
    for (int e = threadIdx.x; e < m * r; e += blockDim.x) S1[(e / r) * kPU + e % r] = MA[e];
    __syncthreads();
    tile_mm4(S1, kPU, false, OR, kPU, false, m, r, r, [&](int i, int j, float v) { S2[i * kPU + j] = v; });
    __syncthreads();
    tile_mm4(Ln, kPU, true, S2, kPU, false, r, r, m, [&](int i, int j, float v) { S1[i * kPU + j] = v; });
    __syncthreads();
    tile_mm4(Ln, kPU, false, S1, kPU, false, m, r, r,
             [&](int i, int j, float v) { MA[i * r + j] = S2[i * kPU + j] - v; });
    __syncthreads();
    // M_B <- O_L M_B (I - U_Rn U_Rn^T):  T = O_L M_B, Y = T U_Rn, M_B = T - Y U_Rn^T
    for (int e = threadIdx.x; e < r * n; e += blockDim.x) S1[(e / n) * kPG + e % n] = MB[e];
    __syncthreads();
    tile_mm4(OL, kPU, false, S1, kPG, false, r, n, r, [&](int i, int j, float v) { S2[i * kPG + j] = v; });
    __syncthreads();
    tile_mm4(S2, kPG, false, Rn, kPU, false, r, r, n, [&](int i, int j, float v) { S1[i * kPU + j] = v; });
    __syncthreads();
    tile_mm4(S1, kPU, false, Rn, kPU, true, r, n, r,
             [&](int i, int j, float v) { MB[i * n + j] = S2[i * kPG + j] - v; });
    // v_A^T <- v_A^T (O_R)^2, v_B <- (O_L)^2 v_B (entry-wise squares)
    float sa = 0.0f, sb = 0.0f;
    const int j = threadIdx.x;
    if (j < r) {
      for (int l = 0; l < r; ++l) {
        sa = fmaf(vA[l], OR[l * kPU + j] * OR[l * kPU + j], sa);
        sb = fmaf(OL[j * kPU + l] * OL[j * kPU + l], vB[l], sb);
      }
    }
    __syncthreads();
    if (j < r) {
      vA[j] = sa;
      vB[j] = sb;
    }
  }
  // the new bases (and their eigenvalues) become current
  for (int e = threadIdx.x; e < m * r; e += blockDim.x) UL[e] = ULn[e];
  for (int e = threadIdx.x; e < n * r; e += blockDim.x) UR[e] = URn[e];
  for (int j = threadIdx.x; j < r; j += blockDim.x) {
    A.lamL[static_cast<int64_t>(b) * r + j] = A.lamLn[static_cast<int64_t>(b) * r + j];
    A.lamR[static_cast<int64_t>(b) * r + j] = A.lamRn[static_cast<int64_t>(b) * r + j];
  }
}

// ----------------------------------------------------------------- the step
template <typename WT>
__device__ __forceinline__ float c_wload(const WT* p);
template <>
__device__ __forceinline__ float c_wload<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float c_wload<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void c_wstore(float* p, float v) { *p = v; }
__device__ __forceinline__ void c_wstore(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Shared-memory plan of the step (floats): every buffer has 4-row slack so
// the tiles' discarded rows stay inside it.
constexpr int kSG = 0;                         // G, then C          (m x n, pitch kPG)
constexpr int kSUL = kSG + kCMax * kPG;        // U_L                (m x r, pitch kPU)
constexpr int kSUR = kSUL + kCMax * kPU;       // U_R                (n x r)
constexpr int kSGU = kSUR + kCMax * kPU;       // G U_R -> G_A -> N(M_A, v_A) -> U_L N(M, V) + N(M_A, v_A)
constexpr int kSUG = kSGU + kCMax * kPU;       // U_L^T G -> G_B -> N(M_B, v_B)  (r x n, pitch kPG)
constexpr int kSS = kSUG + kCK * kPG;          // S -> N(M, V)       (r x r, pitch kPU)
constexpr int kStepFloats = kSS + kCK * kPU;

template <typename WT, typename GT>
__global__ void __launch_bounds__(kCThreads) k_clean_step(CleanArgs A) {
  extern __shared__ float sm[];
  if (c_flagged(A.status)) return;
  const int b = blockIdx.x;
  const int m = A.m, n = A.n, r = A.r;
  const int64_t mn = static_cast<int64_t>(m) * n;
  const GT* G = static_cast<const GT*>(A.G) + b * mn;
  WT* W = static_cast<WT*>(A.W) + b * mn;
  const float* UL = A.UL + static_cast<int64_t>(b) * m * r;
  const float* UR = A.UR + static_cast<int64_t>(b) * n * r;
  float* M = A.Mm + static_cast<int64_t>(b) * r * r;
  float* V = A.Vm + static_cast<int64_t>(b) * r * r;
  float* MA = A.MA + static_cast<int64_t>(b) * m * r;
  float* MB = A.MB + static_cast<int64_t>(b) * r * n;
  float* vA = A.vA + static_cast<int64_t>(b) * r;
  float* vB = A.vB + static_cast<int64_t>(b) * r;
  float* vC = A.vC + b;
  float* Gs = sm + kSG;
  float* ULs = sm + kSUL;
  float* URs = sm + kSUR;
  float* GU = sm + kSGU;
  float* UG = sm + kSUG;
  float* Ss = sm + kSS;
  __shared__ float red[kCThreads / 32];
  bool bad = false;
  for (int e = threadIdx.x; e < mn; e += blockDim.x) {
    const float g = c_gload<GT>(G + e);
    bad |= !isfinite(g);
    Gs[(e / n) * kPG + e % n] = g;
  }
  for (int e = threadIdx.x; e < m * r; e += blockDim.x) ULs[(e / r) * kPU + e % r] = UL[e];
  for (int e = threadIdx.x; e < n * r; e += blockDim.x) URs[(e / r) * kPU + e % r] = UR[e];
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) atomicOr(A.status, kStNonfiniteInput);
    return;
  }
  // G U_R (m x r) and U_L^T G (r x n)
  tile_mm4(Gs, kPG, false, URs, kPU, false, m, r, n, [&](int i, int j, float v) { GU[i * kPU + j] = v; });
  tile_mm4(ULs, kPU, true, Gs, kPG, false, r, n, m, [&](int i, int j, float v) { UG[i * kPG + j] = v; });
  __syncthreads();
  // S = U_L^T (G U_R)
  tile_mm4(ULs, kPU, true, GU, kPU, false, r, r, m, [&](int i, int j, float v) { Ss[i * kPU + j] = v; });
  __syncthreads();
  // G_B = U_L^T G - S U_R^T (in place)
  tile_mm4(Ss, kPU, false, URs, kPU, true, r, n, r, [&](int i, int j, float v) { UG[i * kPG + j] -= v; });
  __syncthreads();
  // C = (I - U_L U_L^T) G (I - U_R U_R^T) = G - U_L G_B - (G U_R) U_R^T, in place;
  // both products hand each element to the same thread, which also sums ||C||^2
  tile_mm4(ULs, kPU, false, UG, kPG, false, m, n, r, [&](int i, int j, float v) { Gs[i * kPG + j] -= v; });
  float sc = 0.0f;
  tile_mm4(GU, kPU, false, URs, kPU, true, m, n, r, [&](int i, int j, float v) {
    const float c = Gs[i * kPG + j] - v;
    Gs[i * kPG + j] = c;
    sc = fmaf(c, c, sc);
  });
  __syncthreads();
  // G_A = G U_R - U_L S (in place)
  tile_mm4(ULs, kPU, false, Ss, kPU, false, m, r, r, [&](int i, int j, float v) { GU[i * kPU + j] -= v; });
  __syncthreads();
  // moments (Table 1)
  const float b1 = A.beta1, b2 = A.beta2;
  for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
    const float s = Ss[(e / r) * kPU + e % r];
    M[e] = fmaf(b1, M[e], (1.0f - b1) * s);
    V[e] = fmaf(b2, V[e], (1.0f - b2) * s * s);
  }
  for (int e = threadIdx.x; e < m * r; e += blockDim.x)
    MA[e] = fmaf(b1, MA[e], (1.0f - b1) * GU[(e / r) * kPU + e % r]);
  for (int e = threadIdx.x; e < r * n; e += blockDim.x)
    MB[e] = fmaf(b1, MB[e], (1.0f - b1) * UG[(e / n) * kPG + e % n]);
  for (int j = threadIdx.x; j < r; j += blockDim.x) {
    float sa = 0.0f, sb = 0.0f;
    for (int i = 0; i < m; ++i) sa = fmaf(GU[i * kPU + j], GU[i * kPU + j], sa);
    for (int q = 0; q < n; ++q) sb = fmaf(UG[j * kPG + q], UG[j * kPG + q], sb);
    vA[j] = fmaf(b2, vA[j], (1.0f - b2) * sa);
    vB[j] = fmaf(b2, vB[j], (1.0f - b2) * sb);
  }
  const float cnorm2 = c_block_sum(sc, red);
  if (threadIdx.x == 0) *vC = fmaf(b2, *vC, (1.0f - b2) * cnorm2);
  __syncthreads();
  // normalised blocks with both bias corrections, in place
  const float bc1 = A.bc1, bc2 = A.bc2, eps = A.eps;
  for (int e = threadIdx.x; e < r * r; e += blockDim.x)
    Ss[(e / r) * kPU + e % r] = (M[e] * bc1) / (sqrtf(V[e] * bc2) + eps);
  for (int e = threadIdx.x; e < m * r; e += blockDim.x)
    GU[(e / r) * kPU + e % r] = (MA[e] * bc1) / (sqrtf(vA[e % r] * bc2) + eps);
  for (int e = threadIdx.x; e < r * n; e += blockDim.x)
    UG[(e / n) * kPG + e % n] = (MB[e] * bc1) / (sqrtf(vB[e / n] * bc2) + eps);
  const float cden = 1.0f / (sqrtf(*vC * bc2) + eps);
  __syncthreads();
  // U_L N(M, V) + N(M_A, v_A), in place
  tile_mm4(ULs, kPU, false, Ss, kPU, false, m, r, r, [&](int i, int j, float v) { GU[i * kPU + j] += v; });
  __syncthreads();
  // G~ = C cden + (U_L N(M, V) + N(M_A, v_A)) U_R^T + U_L N(M_B, v_B), folded
  // into W; both products hand each element to the same thread
  tile_mm4(GU, kPU, false, URs, kPU, true, m, n, r, [&](int i, int j, float v) {
    Gs[i * kPG + j] = fmaf(Gs[i * kPG + j], cden, v);
  });
  tile_mm4(ULs, kPU, false, UG, kPG, false, m, n, r, [&](int i, int j, float v) {
    const float g = Gs[i * kPG + j] + v;
    const int64_t e = static_cast<int64_t>(i) * n + j;
    const float w = fmaf(-A.alr, g, A.decay * c_wload<WT>(W + e));
    bad |= !isfinite(w);
    c_wstore(W + e, w);
  });
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(A.status, kStNonfiniteUpdate);
}

// reset: every moment zero (the bases are written by the first refresh)
__global__ void k_clean_reset(CleanArgs A) {
  const int b = blockIdx.x;
  const int m = A.m, n = A.n, r = A.r;
  for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
    A.Mm[static_cast<int64_t>(b) * r * r + e] = 0.0f;
    A.Vm[static_cast<int64_t>(b) * r * r + e] = 0.0f;
  }
  for (int e = threadIdx.x; e < m * r; e += blockDim.x) A.MA[static_cast<int64_t>(b) * m * r + e] = 0.0f;
  for (int e = threadIdx.x; e < r * n; e += blockDim.x) A.MB[static_cast<int64_t>(b) * r * n + e] = 0.0f;
  for (int j = threadIdx.x; j < r; j += blockDim.x) {
    A.vA[static_cast<int64_t>(b) * r + j] = 0.0f;
    A.vB[static_cast<int64_t>(b) * r + j] = 0.0f;
  }
  if (threadIdx.x == 0) A.vC[b] = 0.0f;
}

constexpr int kCRefreshSmem = kRefreshFloats * 4;
constexpr int kCRotateSmem = kRotateFloats * 4;
constexpr int kCStepSmem = kStepFloats * 4;

static cudaError_t clean_attributes() {
  static PerDevice pd;
  return once_per_device(pd, [](int) {
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(k_clean_refresh<float>, at, kCRefreshSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_refresh<__nv_bfloat16>, at, kCRefreshSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_rotate, at, kCRotateSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_step<float, float>, at, kCStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_step<float, __nv_bfloat16>, at, kCStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_step<__nv_bfloat16, float>, at, kCStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_clean_step<__nv_bfloat16, __nv_bfloat16>, at, kCStepSmem);
    return e;
  });
}

cudaError_t launch_clean_refresh(const CleanArgs& A, cudaStream_t st) {
  cudaError_t e = clean_attributes();
  if (e != cudaSuccess) return e;
  if (A.g_bf16)
    k_clean_refresh<__nv_bfloat16><<<2 * A.batch, kCThreads, kCRefreshSmem, st>>>(A);
  else
    k_clean_refresh<float><<<2 * A.batch, kCThreads, kCRefreshSmem, st>>>(A);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_clean_rotate<<<A.batch, kCThreads, kCRotateSmem, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_clean_step(const CleanArgs& A, cudaStream_t st) {
  cudaError_t e = clean_attributes();
  if (e != cudaSuccess) return e;
  if (A.w_bf16 && A.g_bf16)
    k_clean_step<__nv_bfloat16, __nv_bfloat16><<<A.batch, kCThreads, kCStepSmem, st>>>(A);
  else if (A.w_bf16)
    k_clean_step<__nv_bfloat16, float><<<A.batch, kCThreads, kCStepSmem, st>>>(A);
  else if (A.g_bf16)
    k_clean_step<float, __nv_bfloat16><<<A.batch, kCThreads, kCStepSmem, st>>>(A);
  else
    k_clean_step<float, float><<<A.batch, kCThreads, kCStepSmem, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_clean_reset(const CleanArgs& A, cudaStream_t st) {
  k_clean_reset<<<A.batch, 256, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace okls

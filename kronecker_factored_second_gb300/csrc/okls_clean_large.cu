// Clean for shapes past one CTA's shared memory: m, n up to 16384 and
// r + p <= 544 (sm_103a).
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching": Algorithm 1, Eqn. (8), Appendix A Algorithm 3, Eqns. (10)-(16),
// Table 1 -- the same method as the one-CTA kernels, restated for tall
// operands.  Every product with a dimension that grows with m or n is a
// batched fp32 GEMM (`k_cl_gemm`: 128 x 128 tiles, 8 x 8 per thread,
// double-buffered slices in shared memory); only k x k work (k = r + p) stays in
// one CTA per matrix: the Cholesky factors and inverses of the thin QRs and
// of Omega^T Y_nu, the norm estimate for nu, and the Jacobi eigensolve of
// Z^T Z that yields the thin SVD (past k = 128 the logged-rotation solver of
// okls_eig.cu, whose rotations of V spread over many CTAs).  The thin QRs are Cholesky-QR applied four
// times, a pass shifted where its factorisation breaks down (the
// power-iterated sketch is ill-conditioned), so they reduce to Gram
// products, k x k factorisations and products again.
#include <cuda_bf16.h>

#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

// ---------------------------------------------------------------- the GEMM
// 128 x 128 output tile per CTA, K in slices of 16, 256 threads with 8 x 8
// outputs each (two 4-row by two 4-column groups, so that a warp's float4
// reads of the staged slices are conflict-free); the next slice is fetched
// into registers while the current one is multiplied (double-buffered shared
// memory, one barrier per slice).  A thread fetches 8 consecutive elements of
// each operand per slice, as 16-byte vectors where the layout allows.
constexpr int kGM = 128;  // output tile edge
constexpr int kGK = 16;   // K per slice

template <typename T>
__device__ __forceinline__ float cl_ld(const T* p);
template <>
__device__ __forceinline__ float cl_ld<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float cl_ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// 8 consecutive elements at p (16-byte aligned for the vector forms)
__device__ __forceinline__ void cl_ld8(const float* p, float v[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void cl_ld8(const __nv_bfloat16* p, float v[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    v[2 * u] = __uint_as_float(w[u] << 16);
    v[2 * u + 1] = __uint_as_float(w[u] & 0xffff0000u);
  }
}

// The thread's 8 elements of a slice of an operand staged as [k][128]:
// `kmajor` operands are stored K x rows (a slice row is 128 contiguous
// entries: the thread takes 8 of one k), the others rows x K (the thread
// takes 8 consecutive k of one row).  Out-of-range elements read as 0;
// `vec` says 16-byte loads are aligned for this operand.
template <typename T>
__device__ __forceinline__ void cl_fetch(const T* X, bool kmajor, bool vec, int64_t ld, int row0, int rows, int k0,
                                         int K, float v[8], int& kk, int& i0) {
  const int t = threadIdx.x;
  if (kmajor) {
    kk = t >> 4;
    i0 = (t & 15) * 8;
    const int gk = k0 + kk, gi = row0 + i0;
    const T* p = X + static_cast<int64_t>(gk) * ld + gi;
    if (vec && gk < K && gi + 8 <= rows) {
      cl_ld8(p, v);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (gk < K && gi + u < rows) ? cl_ld<T>(p + u) : 0.0f;
    }
  } else {
    i0 = t >> 1;
    kk = (t & 1) * 8;
    const int gi = row0 + i0, gk = k0 + kk;
    const T* p = X + static_cast<int64_t>(gi) * ld + gk;
    if (vec && gi < rows && gk + 8 <= K) {
      cl_ld8(p, v);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (gi < rows && gk + u < K) ? cl_ld<T>(p + u) : 0.0f;
    }
  }
}

__device__ __forceinline__ void cl_stage(float (*S)[kGM], bool kmajor, const float v[8], int kk, int i0) {
  if (kmajor) {
    *reinterpret_cast<float4*>(&S[kk][i0]) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(&S[kk][i0 + 4]) = make_float4(v[4], v[5], v[6], v[7]);
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u) S[kk + u][i0] = v[u];
  }
}

// C[b] = alpha op(A[b]) op(B[b]) + beta_b C[b], beta_b = beta_dev ? beta_dev[b] : beta.
// A is M x K (lda), or K x M when ta; B is K x N (ldb), or N x K when tb.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_cl_gemm(ClGemm g) {
  __shared__ __align__(16) float As[2][kGK][kGM];
  __shared__ __align__(16) float Bs[2][kGK][kGM];
  // a GEMM that writes state is skipped once an earlier stage has flagged
  if (g.status_guard &&
      __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(g.status_guard) != 0u))
    return;
  const int b = blockIdx.z;
  const TA* A = static_cast<const TA*>(g.A) + static_cast<int64_t>(b) * g.sA;
  const TB* B = static_cast<const TB*>(g.B) + static_cast<int64_t>(b) * g.sB;
  float* C = g.C + static_cast<int64_t>(b) * g.sC;
  const int m0 = blockIdx.y * kGM, n0 = blockIdx.x * kGM;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // A is staged [k][m]: k-major when stored K x M (ta); B is staged [k][n]:
  // k-major when stored K x N (not tb)
  const bool a_kmaj = g.ta != 0, b_kmaj = g.tb == 0;
  float acc[8][8] = {};
  float va[8], vb[8];
  int akk, ai0, bkk, bi0;
  cl_fetch<TA>(A, a_kmaj, g.a_vec, g.lda, m0, g.M, 0, g.K, va, akk, ai0);
  cl_fetch<TB>(B, b_kmaj, g.b_vec, g.ldb, n0, g.N, 0, g.K, vb, bkk, bi0);
  cl_stage(As[0], a_kmaj, va, akk, ai0);
  cl_stage(Bs[0], b_kmaj, vb, bkk, bi0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < g.K; k0 += kGK) {
    const bool more = k0 + kGK < g.K;
    if (more) {
      cl_fetch<TA>(A, a_kmaj, g.a_vec, g.lda, m0, g.M, k0 + kGK, g.K, va, akk, ai0);
      cl_fetch<TB>(B, b_kmaj, g.b_vec, g.ldb, n0, g.N, k0 + kGK, g.K, vb, bkk, bi0);
    }
#pragma unroll
    for (int kk = 0; kk < kGK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    if (more) {
      cl_stage(As[buf ^ 1], a_kmaj, va, akk, ai0);
      cl_stage(Bs[buf ^ 1], b_kmaj, vb, bkk, bi0);
    }
    __syncthreads();
    buf ^= 1;
  }
  const float beta = g.beta_dev ? g.beta_dev[b] : g.beta;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int gm = m0 + (u < 4 ? ty * 4 + u : 64 + ty * 4 + u - 4);
    if (gm >= g.M) continue;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int gn = n0 + (v < 4 ? tx * 4 + v : 64 + tx * 4 + v - 4);
      if (gn >= g.N) continue;
      float* c = C + static_cast<int64_t>(gm) * g.ldc + gn;
      *c = beta == 0.0f ? g.alpha * acc[u][v] : fmaf(g.alpha, acc[u][v], beta * *c);
    }
  }
}

// 16-byte loads of 8 elements need the base, the leading dimension and the
// batch stride to keep every run of 8 on a 16-byte boundary
static int cl_vec_ok(const void* p, int bf16, int64_t ld, int64_t stride) {
  const int64_t q = bf16 ? 8 : 4;  // elements per 16 bytes
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ld % q == 0 && stride % q == 0;
}

cudaError_t launch_cl_gemm(const ClGemm& g0, cudaStream_t st) {
  if (g0.M <= 0 || g0.N <= 0 || g0.batch <= 0) return cudaSuccess;
  ClGemm g = g0;
  g.a_vec = cl_vec_ok(g.A, g.a_bf16, g.lda, g.sA);
  g.b_vec = cl_vec_ok(g.B, g.b_bf16, g.ldb, g.sB);
  if (t3_gemm_eligible(g)) return launch_t3_gemm(g, st);
  const dim3 grid((g.N + kGM - 1) / kGM, (g.M + kGM - 1) / kGM, g.batch);
  if (g.a_bf16 && g.b_bf16)
    k_cl_gemm<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(g);
  else if (g.a_bf16)
    k_cl_gemm<__nv_bfloat16, float><<<grid, 256, 0, st>>>(g);
  else if (g.b_bf16)
    k_cl_gemm<float, __nv_bfloat16><<<grid, 256, 0, st>>>(g);
  else
    k_cl_gemm<float, float><<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

// ------------------------------------------------------------- k x k kernels
// Up to k = kLK the two k x k matrices of these kernels live in shared
// memory; past it (k <= kClMaxK) in a per-matrix workspace slice of
// 2 (k + 1)^2 floats, which stays in L2 -- the same code, a slower access.
constexpr int kLK = 128;
constexpr int kLP = kLK + 1;        // odd pitch of the staged k x k matrices
constexpr int kLThreads = 256;
constexpr int kLWide = 1024;  // the packed Cholesky: more of a step's work in flight
constexpr int kLVec = 2 * kClMaxK;  // floats: vectors / rotation parameters
constexpr int kLInts = 2 * kClMaxK; // ints: pairs, then ranks
constexpr int kLHead = kLVec + kLInts;
constexpr int kLSmallSmem = (kLHead + 2 * kLK * kLP) * 4;
// up to here the k x k matrix of the packed Cholesky kernel fits shared
// memory as a packed triangle
constexpr int kPackMaxK = 330;

struct KkStore {
  float* a;
  float* b;
  int ld;
};

__device__ __forceinline__ KkStore kk_store(float* sm, float* scratch, int k) {
  if (k <= kLK) return {sm + kLHead, sm + kLHead + kLK * kLP, kLP};
  // (k + 1) rows of pitch k + 1: the Jacobi iteration pads an odd k by one
  float* g = scratch + static_cast<int64_t>(blockIdx.x) * 2 * (k + 1) * (k + 1);
  return {g, g + static_cast<int64_t>(k + 1) * (k + 1), k + 1};
}

inline int kk_smem(int k) { return k <= kLK ? kLSmallSmem : kLHead * 4; }

__device__ __forceinline__ bool cl_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

__device__ __forceinline__ float cl_block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
  return s;
}

// Cholesky factor of the symmetric part of a k x k Gram matrix and the
// inverse of its upper factor R = L^T: Rinv = L^-T, so that X Rinv has
// orthonormal columns when Gram = X^T X.  With `adaptive` a breakdown (a
// pivot that is not positive: the panel's condition number squared has
// passed 2^24) restarts the factorisation with the diagonal shifted by
// 11 (k + sqrt(d)) 2^-24 trace(Gram), above the rounding error of the Gram
// product -- shifted Cholesky-QR, which trades a well-conditioned factor for
// a partial orthogonalisation that the next pass completes.  A breakdown
// that remains raises kStNonfiniteIter.
__global__ void __launch_bounds__(kLThreads) k_cl_chol_inv(const float* Gram, float* Rinv, int k, int d, int adaptive,
                                                           float* scratch, uint32_t* status) {
  extern __shared__ float sm[];
  __shared__ float red[kLThreads / 32];
  __shared__ float piv;
  const int b = blockIdx.x;
  const float* Gb = Gram + static_cast<int64_t>(b) * k * k;
  float* Rb = Rinv + static_cast<int64_t>(b) * k * k;
  const KkStore ks = kk_store(sm, scratch, k);
  const int ld = ks.ld;
  float* Ls = ks.a;  // k x k, lower triangle used
  float* Xs = ks.b;  // L^-1, column by column
  float tr = 0.0f;
  for (int e = threadIdx.x; e < k * k; e += blockDim.x)
    if (e / k == e % k) tr += Gb[e];
  tr = cl_block_sum(tr, red);
  bool bad = false;
  for (int attempt = 0; attempt < (adaptive ? 2 : 1); ++attempt) {
    const float sh = attempt == 0 ? 0.0f : 11.0f * (k + sqrtf(static_cast<float>(d))) * 5.9604645e-8f * tr;
    for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
      const int i = e / k, j = e % k;
      Ls[i * ld + j] = 0.5f * (Gb[i * k + j] + Gb[j * k + i]) + (i == j ? sh : 0.0f);
    }
    __syncthreads();
    bad = false;
    for (int j = 0; j < k; ++j) {
      if (threadIdx.x == 0) {
        const float djj = Ls[j * ld + j];
        piv = djj > 0.0f ? sqrtf(djj) : 0.0f;
      }
      __syncthreads();
      const float cj = piv;
      if (!(cj > 0.0f)) bad = true;
      for (int i = j + threadIdx.x; i < k; i += blockDim.x)
        Ls[i * ld + j] = i == j ? cj : (cj > 0.0f ? Ls[i * ld + j] / cj : 0.0f);
      __syncthreads();
      const int w = k - j - 1;
      for (int e = threadIdx.x; e < w * w; e += blockDim.x) {
        const int i = j + 1 + e / w, l = j + 1 + e % w;
        if (l <= i) Ls[i * ld + l] = fmaf(-Ls[i * ld + j], Ls[l * ld + j], Ls[i * ld + l]);
      }
      __syncthreads();
    }
    if (!__syncthreads_or(bad)) break;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) atomicOr(status, kStNonfiniteIter);
    return;
  }
  // column c of L^-1 by forward substitution (one thread per column)
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    for (int i = 0; i < c; ++i) Xs[i * ld + c] = 0.0f;
    Xs[c * ld + c] = 1.0f / Ls[c * ld + c];
    for (int i = c + 1; i < k; ++i) {
      float v = 0.0f;
      for (int l = c; l < i; ++l) v = fmaf(Ls[i * ld + l], Xs[l * ld + c], v);
      Xs[i * ld + c] = -v / Ls[i * ld + i];
    }
  }
  __syncthreads();
  // Rinv = (L^-1)^T
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    Rb[e] = Xs[j * ld + i];
  }
}

// The same factorisation for 128 < k <= kPackMaxK with L as a packed lower
// triangle in shared memory; each thread forward-substitutes a column of
// L^-1 straight into the matching row of Rinv = L^-T.
__device__ __forceinline__ int pl_idx(int i, int j) { return i * (i + 1) / 2 + j; }  // i >= j

__global__ void __launch_bounds__(kLWide) k_cl_chol_inv_packed(const float* Gram, float* Rinv, int k, int d,
                                                                  int adaptive, uint32_t* status) {
  extern __shared__ float sm[];
  __shared__ float red[kLWide / 32];
  __shared__ float piv;
  const int b = blockIdx.x;
  const float* Gb = Gram + static_cast<int64_t>(b) * k * k;
  float* Rb = Rinv + static_cast<int64_t>(b) * k * k;
  float* Ls = sm + kLHead;
  float tr = 0.0f;
  for (int i = threadIdx.x; i < k; i += blockDim.x) tr += Gb[i * k + i];
  tr = cl_block_sum(tr, red);
  bool bad = false;
  for (int attempt = 0; attempt < (adaptive ? 2 : 1); ++attempt) {
    const float sh = attempt == 0 ? 0.0f : 11.0f * (k + sqrtf(static_cast<float>(d))) * 5.9604645e-8f * tr;
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      for (int j = 0; j <= i; ++j) Ls[pl_idx(i, j)] = 0.5f * (Gb[i * k + j] + Gb[j * k + i]) + (i == j ? sh : 0.0f);
    __syncthreads();
    bad = false;
    for (int j = 0; j < k; ++j) {
      if (threadIdx.x == 0) {
        const float djj = Ls[pl_idx(j, j)];
        piv = djj > 0.0f ? sqrtf(djj) : 0.0f;
      }
      __syncthreads();
      const float cj = piv;
      if (!(cj > 0.0f)) bad = true;
      for (int i = j + threadIdx.x; i < k; i += blockDim.x)
        Ls[pl_idx(i, j)] = i == j ? cj : (cj > 0.0f ? Ls[pl_idx(i, j)] / cj : 0.0f);
      __syncthreads();
      const int w = k - j - 1;
      for (int e = threadIdx.x; e < w * w; e += blockDim.x) {
        const int i = j + 1 + e / w, l = j + 1 + e % w;
        if (l <= i) Ls[pl_idx(i, l)] = fmaf(-Ls[pl_idx(i, j)], Ls[pl_idx(l, j)], Ls[pl_idx(i, l)]);
      }
      __syncthreads();
    }
    if (!__syncthreads_or(bad)) break;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) atomicOr(status, kStNonfiniteIter);
    return;
  }
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    float* x = Rb + static_cast<int64_t>(c) * k;  // row c of Rinv = column c of L^-1
    for (int i = 0; i < c; ++i) x[i] = 0.0f;
    x[c] = 1.0f / Ls[pl_idx(c, c)];
    for (int i = c + 1; i < k; ++i) {
      float v = 0.0f;
      for (int l = c; l < i; ++l) v = fmaf(Ls[pl_idx(i, l)], x[l], v);
      x[i] = -v / Ls[pl_idx(i, i)];
    }
  }
}

inline int packed_chol_smem(int k) { return (kLHead + k * (k + 1) / 2) * 4; }

// nu = spacing of binary32 numbers at ||Y||_2, ||Y||_2^2 the largest
// eigenvalue of the Gram matrix Y^T Y (60 power steps; every warp takes
// rows of the product).
__global__ void __launch_bounds__(kLThreads) k_cl_norm(const float* Gram, float* nu, int k, float* scratch) {
  extern __shared__ float sm[];
  __shared__ float red[kLThreads / 32];
  const int b = blockIdx.x;
  const float* Gb = Gram + static_cast<int64_t>(b) * k * k;
  const KkStore ks = kk_store(sm, scratch, k);
  const int ld = ks.ld;
  float* As = ks.a;
  float* v = sm;  // 2 k: the iterate and its image
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) As[(e / k) * ld + e % k] = Gb[e];
  for (int j = threadIdx.x; j < k; j += blockDim.x) v[j] = 1.0f;
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float nrm = 0.0f;
  for (int it = 0; it < 60; ++it) {
    float s2 = 0.0f;
    for (int i = w; i < k; i += nw) {
      float s = 0.0f;
      for (int j = lane; j < k; j += 32) s = fmaf(As[static_cast<int64_t>(i) * ld + j], v[j], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) v[kClMaxK + i] = s;
      s2 = fmaf(s, s, s2);
    }
    // s2 is the same on every lane of a warp: count it once per warp
    nrm = sqrtf(cl_block_sum(lane == 0 ? s2 : 0.0f, red));
    for (int i = threadIdx.x; i < k; i += blockDim.x) v[i] = nrm > 0.0f ? v[kClMaxK + i] / nrm : 0.0f;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float yn = sqrtf(nrm);
    nu[b] = yn > 0.0f ? ldexpf(1.0f, ilogbf(yn) - 23) : 0.0f;
  }
}

// Thin SVD of Z from the eigen-decomposition of Z^T Z = V Sigma^2 V^T (cyclic
// Jacobi in shared memory).  Writes WU (k x r) with U = Z WU: column c of WU
// is s_c v_j / sigma_j for the eigenpair j of rank c (decreasing Sigma^2),
// s_c = +-1 aligning U's column with the previous basis (P = Z^T U_prev,
// k x r; null at the first refresh); and Lambda_c = max(0, sigma_j^2 - nu).
__global__ void __launch_bounds__(kLThreads) k_cl_svd(const float* Gram, const float* P, const float* nu, float* WU,
                                                      float* lam, int k, int r, int max_sweeps, float tol2,
                                                      float* scratch, const uint32_t* status) {
  extern __shared__ float sm[];
  __shared__ float red[kLThreads / 32];
  if (cl_flagged(status)) return;
  const int b = blockIdx.x;
  const float* Gb = Gram + static_cast<int64_t>(b) * k * k;
  const KkStore ks = kk_store(sm, scratch, k);
  const int ld = ks.ld;
  float* As = ks.a;
  float* Vs = ks.b;
  float* cs = sm;                                  // 2 per pair
  int* pr = reinterpret_cast<int*>(sm + kLVec);    // 2 per pair, then ranks
  const int dp = k + (k & 1), np = dp / 2;
  for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
    const int i = e / dp, j = e % dp;
    As[i * ld + j] = (i < k && j < k) ? 0.5f * (Gb[i * k + j] + Gb[j * k + i]) : 0.0f;
    Vs[i * ld + j] = i == j ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    float off = 0.0f, dg = 0.0f;
    for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
      const int i = e / dp, j = e % dp;
      const float v = As[i * ld + j];
      if (i == j)
        dg = fmaf(v, v, dg);
      else
        off = fmaf(v, v, off);
    }
    const float offs = cl_block_sum(off, red);
    const float dgs = cl_block_sum(dg, red);
    if (!(offs > tol2 * dgs)) break;
    for (int rd = 0; rd < dp - 1; ++rd) {
      for (int q = threadIdx.x; q < np; q += blockDim.x) {
        auto idx = [&](int pos) { return pos == 0 ? 0 : 1 + (pos - 1 + rd) % (dp - 1); };
        int pp = idx(q), qq = idx(dp - 1 - q);
        if (pp > qq) {
          const int x = pp;
          pp = qq;
          qq = x;
        }
        const float apq = As[pp * ld + qq];
        const float app = As[pp * ld + pp], aqq = As[qq * ld + qq];
        float c = 1.0f, sn = 0.0f;
        // threshold Jacobi: a pair already below tol2 / k of its diagonal is
        // left alone (when every pair is, the sweep's stopping rule holds)
        if (apq * apq > tol2 / static_cast<float>(k) * fabsf(app * aqq)) {
          const float th = (aqq - app) / (2.0f * apq);
          const float t = copysignf(1.0f, th) / (fabsf(th) + sqrtf(fmaf(th, th, 1.0f)));
          c = rsqrtf(fmaf(t, t, 1.0f));
          sn = t * c;
        }
        cs[2 * q] = c;
        cs[2 * q + 1] = sn;
        pr[2 * q] = pp;
        pr[2 * q + 1] = qq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * dp; e += blockDim.x) {
        const int q = e / dp, j = e % dp;
        const float c = cs[2 * q], sn = cs[2 * q + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * q], qq = pr[2 * q + 1];
        const float ap = As[pp * ld + j], aq = As[qq * ld + j];
        As[pp * ld + j] = c * ap - sn * aq;
        As[qq * ld + j] = sn * ap + c * aq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * dp; e += blockDim.x) {
        const int q = e / dp, i = e % dp;
        const float c = cs[2 * q], sn = cs[2 * q + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * q], qq = pr[2 * q + 1];
        const float ap = As[i * ld + pp], aq = As[i * ld + qq];
        As[i * ld + pp] = c * ap - sn * aq;
        As[i * ld + qq] = sn * ap + c * aq;
        const float vp = Vs[i * ld + pp], vq = Vs[i * ld + qq];
        Vs[i * ld + pp] = c * vp - sn * vq;
        Vs[i * ld + qq] = sn * vp + c * vq;
      }
      __syncthreads();
    }
  }
  // ranks by decreasing Sigma^2 (ties by index)
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const float lj = As[j * ld + j];
    int rank = 0;
    for (int i = 0; i < k; ++i) {
      const float li = As[i * ld + i];
      rank += (li > lj) || (li == lj && i < j);
    }
    pr[j] = rank;
  }
  __syncthreads();
  // nu null: plain eigenvectors (no 1/sigma scaling) and eigenvalues
  const bool unit = nu == nullptr;
  const float nub = unit ? 0.0f : nu[b];
  float* W = WU + static_cast<int64_t>(b) * k * r;
  const float* Pb = P ? P + static_cast<int64_t>(b) * k * r : nullptr;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const int c = pr[j];
    if (c >= r) continue;
    const float s2 = As[j * ld + j];
    const float inv = unit ? 1.0f : (s2 > 0.0f ? rsqrtf(s2) : 0.0f);
    float sg = 1.0f;
    if (Pb) {
      float dot = 0.0f;
      for (int l = 0; l < k; ++l) dot = fmaf(Vs[l * ld + j], Pb[l * r + c], dot);
      sg = dot < 0.0f ? -1.0f : 1.0f;
    }
    for (int l = 0; l < k; ++l) W[l * r + c] = sg * inv * Vs[l * ld + j];
    if (lam) lam[static_cast<int64_t>(b) * r + c] = unit ? s2 : fmaxf(0.0f, s2 - nub);
  }
}


// ------------------------------------------------------- element-wise kernels
// Omega = [U_prev, Psi] (warm) or Psi (cold) for one side: rows row0.. of the
// noise block, d rows, k columns.
__global__ void k_cl_omega(const float* Uprev, const float* noise, float* Om, int d, int k, int r, int mn, int row0,
                           int warm, int64_t om_stride) {
  const int b = blockIdx.y;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < static_cast<int64_t>(d) * k;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(e / k), j = static_cast<int>(e % k);
    const float* nz = noise + (static_cast<int64_t>(b) * mn + row0 + i) * k;
    float v;
    if (warm)
      v = j < r ? Uprev[(static_cast<int64_t>(b) * d + i) * r + j] : nz[j - r];
    else
      v = nz[j];
    Om[b * om_stride + e] = v;
  }
}

// X (rows x cols, batch-strided) += coef[b] * Y; or X[i][j] *= rowscale[b][i]
__global__ void k_cl_axpy(float* X, const float* Y, const float* coef, int64_t elems, int64_t stride) {
  const int b = blockIdx.y;
  const float c = coef[b];
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < elems;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    X[b * stride + e] = fmaf(c, Y[b * stride + e], X[b * stride + e]);
}

__global__ void k_cl_rowscale(float* X, const float* scale, int rows, int cols, int64_t stride, int scale_stride) {
  const int b = blockIdx.y;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < static_cast<int64_t>(rows) * cols;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    X[b * stride + e] *= scale[static_cast<int64_t>(b) * scale_stride + e / cols];
}

template <typename GT>
__global__ void k_cl_prep(const GT* G, float* Cb, int64_t mn, uint32_t* status) {
  const int b = blockIdx.y;
  bool bad = false;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float g = cl_ld<GT>(G + b * mn + e);
    bad |= !isfinite(g);
    Cb[b * mn + e] = g;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kStNonfiniteInput);
}

// fixed-slot partial sums of squares (kClParts blocks per matrix, summed in
// order by k_cl_moments)
__global__ void __launch_bounds__(256) k_cl_sumsq(const float* X, int64_t elems, float* part) {
  __shared__ float red[8];
  const int b = blockIdx.y;
  float s = 0.0f;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < elems;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = X[b * elems + e];
    s = fmaf(v, v, s);
  }
  s = cl_block_sum(s, red);
  if (threadIdx.x == 0) part[static_cast<int64_t>(b) * kClParts + blockIdx.x] = s;
}

// One CTA per matrix: Main moments and N(M, V); the pooled second moments of
// blocks A, B and C; the C normaliser.
__global__ void __launch_bounds__(256) k_cl_moments(ClLarge L) {
  if (cl_flagged(L.status)) return;
  const int b = blockIdx.x;
  const int m = L.m, n = L.n, r = L.r;
  float* M = L.M + static_cast<int64_t>(b) * r * r;
  float* V = L.V + static_cast<int64_t>(b) * r * r;
  const float* S = L.S + static_cast<int64_t>(b) * r * r;
  float* Nm = L.Nm + static_cast<int64_t>(b) * r * r;
  const float* GA = L.GU + static_cast<int64_t>(b) * m * r;
  const float* GB = L.UG + static_cast<int64_t>(b) * r * n;
  const float b1 = L.beta1, b2 = L.beta2;
  for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
    const float s = S[e];
    const float mm = fmaf(b1, M[e], (1.0f - b1) * s);
    const float vv = fmaf(b2, V[e], (1.0f - b2) * s * s);
    M[e] = mm;
    V[e] = vv;
    Nm[e] = (mm * L.bc1) / (sqrtf(vv * L.bc2) + L.eps);
  }
  // v_A: column sums of G_A^2; v_B: row sums of G_B^2 (a warp per column / row)
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = w; j < r; j += blockDim.x >> 5) {
    float sa = 0.0f, sb = 0.0f;
    for (int i = lane; i < m; i += 32) sa = fmaf(GA[static_cast<int64_t>(i) * r + j], GA[static_cast<int64_t>(i) * r + j], sa);
    for (int i = lane; i < n; i += 32) sb = fmaf(GB[static_cast<int64_t>(j) * n + i], GB[static_cast<int64_t>(j) * n + i], sb);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, o);
      sb += __shfl_xor_sync(0xffffffffu, sb, o);
    }
    if (lane == 0) {
      L.vA[static_cast<int64_t>(b) * r + j] = fmaf(b2, L.vA[static_cast<int64_t>(b) * r + j], (1.0f - b2) * sa);
      L.vB[static_cast<int64_t>(b) * r + j] = fmaf(b2, L.vB[static_cast<int64_t>(b) * r + j], (1.0f - b2) * sb);
    }
  }
  if (threadIdx.x == 0) {
    float c2 = 0.0f;
    for (int i = 0; i < kClParts; ++i) c2 += L.part[static_cast<int64_t>(b) * kClParts + i];
    const float vc = fmaf(b2, L.vC[b], (1.0f - b2) * c2);
    L.vC[b] = vc;
    L.cden[b] = 1.0f / (sqrtf(vc * L.bc2) + L.eps);
  }
}

// Block A and B first moments, then their normalised forms in place of G_A,
// G_B (one index space: m r entries of A, then r n of B).
__global__ void __launch_bounds__(256) k_cl_blocks(ClLarge L) {
  if (cl_flagged(L.status)) return;
  const int b = blockIdx.y;
  const int m = L.m, n = L.n, r = L.r;
  const int64_t na = static_cast<int64_t>(m) * r, nb = static_cast<int64_t>(r) * n;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < na + nb;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (e < na) {
      const int64_t o = b * na + e;
      const float mv = fmaf(L.beta1, L.MA[o], (1.0f - L.beta1) * L.GU[o]);
      L.MA[o] = mv;
      L.GU[o] = (mv * L.bc1) / (sqrtf(L.vA[static_cast<int64_t>(b) * r + e % r] * L.bc2) + L.eps);
    } else {
      const int64_t f = e - na, o = b * nb + f;
      const float mv = fmaf(L.beta1, L.MB[o], (1.0f - L.beta1) * L.UG[o]);
      L.MB[o] = mv;
      L.UG[o] = (mv * L.bc1) / (sqrtf(L.vB[static_cast<int64_t>(b) * r + f / n] * L.bc2) + L.eps);
    }
  }
}

template <typename WT>
__device__ __forceinline__ void cl_st(WT* p, float v);
template <>
__device__ __forceinline__ void cl_st<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void cl_st<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename WT>
__global__ void __launch_bounds__(256) k_cl_update(WT* W, const float* Gt, int64_t mn, float decay, float alr,
                                                   uint32_t* status) {
  if (cl_flagged(status)) return;
  const int b = blockIdx.y;
  bool bad = false;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t o = b * mn + e;
    const float w = fmaf(-alr, Gt[o], decay * cl_ld<WT>(W + o));
    bad |= !isfinite(w);
    cl_st<WT>(W + o, w);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kStNonfiniteUpdate);
}

// v_A^T <- v_A^T (O_R)^2, v_B <- (O_L)^2 v_B (entry-wise squares); one CTA per matrix
__global__ void k_cl_vrot(const float* vA, const float* vB, const float* OL, const float* OR, float* vAn, float* vBn,
                          int r) {
  const int b = blockIdx.x;
  const float* ol = OL + static_cast<int64_t>(b) * r * r;
  const float* orr = OR + static_cast<int64_t>(b) * r * r;
  for (int j = threadIdx.x; j < r; j += blockDim.x) {
    float sa = 0.0f, sb = 0.0f;
    for (int l = 0; l < r; ++l) {
      sa = fmaf(vA[static_cast<int64_t>(b) * r + l], orr[l * r + j] * orr[l * r + j], sa);
      sb = fmaf(ol[j * r + l] * ol[j * r + l], vB[static_cast<int64_t>(b) * r + l], sb);
    }
    vAn[static_cast<int64_t>(b) * r + j] = sa;
    vBn[static_cast<int64_t>(b) * r + j] = sb;
  }
}

// The refreshed bases (and, after a warm refresh, the transported moments)
// become the state -- unless an earlier stage flagged the status word.
__global__ void k_cl_install(ClLarge L) {
  if (cl_flagged(L.status)) return;
  const int b = blockIdx.y;
  const int64_t m = L.m, n = L.n, r = L.r;
  auto copy = [&](float* dst, const float* src, int64_t elems) {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < elems;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
      dst[b * elems + e] = src[b * elems + e];
  };
  copy(L.UL, L.ULn, m * r);
  copy(L.UR, L.URn, n * r);
  copy(L.lamL, L.lamLn, r);
  copy(L.lamR, L.lamRn, r);
  if (L.warm) {
    copy(L.M, L.Mn, r * r);
    copy(L.MA, L.MAn, m * r);
    copy(L.MB, L.MBn, r * n);
    copy(L.vA, L.vAn, r);
    copy(L.vB, L.vBn, r);
  }
}



// ------------------------------------------------------------- orchestration
namespace {

struct ClRun {
  const ClLarge& L;
  cudaStream_t st;
  int* launches;
  cudaError_t err = cudaSuccess;

  // C = alpha op(A) op(B) + beta C over the batch
  void gemm(const void* A, int abf, int ta, int64_t lda, int64_t sA, const void* B, int bbf, int tb, int64_t ldb,
            int64_t sB, float* C, int64_t ldc, int64_t sC, int M, int N, int K, float alpha = 1.0f, float beta = 0.0f,
            const float* beta_dev = nullptr) {
    if (err != cudaSuccess) return;
    ClGemm g{};
    g.A = A;
    g.B = B;
    g.C = C;
    g.a_bf16 = abf;
    g.b_bf16 = bbf;
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
    g.batch = L.batch;
    g.alpha = alpha;
    g.beta = beta;
    g.beta_dev = beta_dev;
    g.status = L.status;
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
  dim3 grid_for(int64_t elems) const {
    const int64_t g = (elems + 255) / 256;
    return dim3(static_cast<unsigned>(g < 256 ? (g > 0 ? g : 1) : 256), static_cast<unsigned>(L.batch));
  }
};

void cl_chol(const ClLarge& L, int k, int d, int adaptive, cudaStream_t st) {
  if (k > kLK && k <= kPackMaxK)
    k_cl_chol_inv_packed<<<L.batch, kLWide, packed_chol_smem(k), st>>>(L.Gram, L.Rinv, k, d, adaptive, L.status);
  else
    k_cl_chol_inv<<<L.batch, kLThreads, kk_smem(k), st>>>(L.Gram, L.Rinv, k, d, adaptive, L.KK, L.status);
}

cudaError_t cl_attributes() {
  static PerDevice pd;
  return once_per_device(pd, [](int) {
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(k_cl_chol_inv, at, kLSmallSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_cl_norm, at, kLSmallSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_cl_svd, at, kLSmallSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_cl_chol_inv_packed, at, packed_chol_smem(kPackMaxK));
    return e;
  });
}

// Thin QR of the batch of d x k panels in `cur`: four Cholesky-QR passes,
// each shifted only where its factorisation breaks down (panels with
// condition numbers up to ~1e6 come out orthonormal); `spare` is a second
// panel buffer.  An even number of passes leaves Q in `cur`.
float* cl_qr(ClRun& R, float* cur, float* spare, int d) {
  const ClLarge& L = R.L;
  const int k = L.k;
  const int64_t sP = static_cast<int64_t>(L.m > L.n ? L.m : L.n) * k, sK = static_cast<int64_t>(k) * k;
  for (int pass = 0; pass < 4; ++pass) {
    R.gemm(cur, 0, 1, k, sP, cur, 0, 0, k, sP, L.Gram, k, sK, k, k, d);
    R.launch([&] { cl_chol(L, k, d, 1, R.st); });
    R.gemm(cur, 0, 0, k, sP, L.Rinv, 0, 0, k, sK, spare, k, sP, d, k, k);
    float* t = cur;
    cur = spare;
    spare = t;
  }
  return cur;
}

// Y = (b2 U Lambda U^T + (1 - b2) G G^T) X on the left side (side 0), or
// with G^T G on the right side; the factor is never formed.
void cl_apply(ClRun& R, int side, const float* X, float* Y) {
  const ClLarge& L = R.L;
  const int m = L.m, n = L.n, r = L.r, k = L.k;
  const int64_t sP = static_cast<int64_t>(m > n ? m : n) * k, mn = static_cast<int64_t>(m) * n;
  const int d = side == 0 ? m : n;
  if (side == 0) {
    R.gemm(L.G, L.g_bf16, 1, n, mn, X, 0, 0, k, sP, L.T1, k, sP, n, k, m);
    R.gemm(L.G, L.g_bf16, 0, n, mn, L.T1, 0, 0, k, sP, Y, k, sP, m, k, n, 1.0f - L.beta2);
  } else {
    R.gemm(L.G, L.g_bf16, 0, n, mn, X, 0, 0, k, sP, L.T1, k, sP, m, k, n);
    R.gemm(L.G, L.g_bf16, 1, n, mn, L.T1, 0, 0, k, sP, Y, k, sP, n, k, m, 1.0f - L.beta2);
  }
  if (L.warm) {
    const float* U = side == 0 ? L.UL : L.UR;
    const float* lam = side == 0 ? L.lamL : L.lamR;
    const int64_t sU = static_cast<int64_t>(d) * r;
    R.gemm(U, 0, 1, r, sU, X, 0, 0, k, sP, L.T1, k, sP, r, k, d);
    R.launch([&] {
      k_cl_rowscale<<<R.grid_for(static_cast<int64_t>(r) * k), 256, 0, R.st>>>(L.T1, lam, r, k, sP, r);
    });
    R.gemm(U, 0, 0, r, sU, L.T1, 0, 0, k, sP, Y, k, sP, d, k, r, L.beta2, 1.0f);
  }
}

// Algorithm 3 for one side: the new basis (d x r) and eigenvalues.
void cl_nystrom(ClRun& R, int side) {
  const ClLarge& L = R.L;
  const int m = L.m, n = L.n, r = L.r, k = L.k;
  const int d = side == 0 ? m : n;
  const int64_t sP = static_cast<int64_t>(m > n ? m : n) * k, sK = static_cast<int64_t>(k) * k;
  const int64_t sU = static_cast<int64_t>(d) * r;
  const float* Uprev = side == 0 ? L.UL : L.UR;
  float* Uout = side == 0 ? L.ULn : L.URn;
  float* lamOut = side == 0 ? L.lamLn : L.lamRn;
  R.launch([&] {
    k_cl_omega<<<R.grid_for(static_cast<int64_t>(d) * k), 256, 0, R.st>>>(Uprev, L.noise, L.Om, d, k, r, m + n,
                                                                          side == 0 ? 0 : m, L.warm, sP);
  });
  // panels: Om, X (QR ping-pong), Y, T1 (apply's temporary)
  float* om = cl_qr(R, L.Om, L.X, d);  // Q in Om
  for (int it = 0; it < L.q; ++it) {
    cl_apply(R, side, om, L.Y);
    om = cl_qr(R, L.Y, L.X, d);  // Q in Y; Om is spent
    float* t = om == L.Y ? L.Om : om;
    if (om == L.Y) {
      // keep the basis out of the Y panel, which the next apply writes
      if (R.err == cudaSuccess)
        R.err = cudaMemcpyAsync(t, L.Y, static_cast<size_t>(L.batch) * sP * 4, cudaMemcpyDeviceToDevice, R.st);
      om = t;
    }
  }
  float* free_panel = om == L.Om ? L.X : L.Om;
  cl_apply(R, side, om, L.Y);
  // nu = eps(||Y||_2); Y_nu = Y + nu Omega
  R.gemm(L.Y, 0, 1, k, sP, L.Y, 0, 0, k, sP, L.Gram, k, sK, k, k, d);
  R.launch([&] { k_cl_norm<<<L.batch, kLThreads, kk_smem(k), R.st>>>(L.Gram, L.nu, k, L.KK); });
  R.launch([&] { k_cl_axpy<<<R.grid_for(static_cast<int64_t>(d) * k), 256, 0, R.st>>>(L.Y, om, L.nu, static_cast<int64_t>(d) * k, sP); });
  // C^T C = (B + B^T)/2, B = Omega^T Y_nu;  Z = Y_nu C^-1
  R.gemm(om, 0, 1, k, sP, L.Y, 0, 0, k, sP, L.Gram, k, sK, k, k, d);
  R.launch([&] { cl_chol(L, k, d, 0, R.st); });
  float* Z = free_panel;
  R.gemm(L.Y, 0, 0, k, sP, L.Rinv, 0, 0, k, sK, Z, k, sP, d, k, k);
  // thin SVD of Z from Z^T Z; signs against the previous basis
  R.gemm(Z, 0, 1, k, sP, Z, 0, 0, k, sP, L.Gram, k, sK, k, k, d);
  if (L.warm) R.gemm(Z, 0, 1, k, sP, Uprev, 0, 0, r, sU, L.P, r, static_cast<int64_t>(k) * r, k, r, d);
  if (k > kLK) {
    EigPlan plan{};
    plan.side[0] = EigSide{L.Gram, L.warm ? L.P : nullptr, L.nu, L.WU, lamOut, L.KK, k, r, L.batch};
    plan.max_sweeps = L.max_sweeps;
    plan.tol2 = L.tol2;
    plan.status = L.status;
    if (R.err == cudaSuccess) R.err = launch_eig_rounds(plan, R.st, R.launches);
  } else {
    R.launch([&] {
      k_cl_svd<<<L.batch, kLThreads, kk_smem(k), R.st>>>(L.Gram, L.warm ? L.P : nullptr, L.nu, L.WU, lamOut, k, r,
                                                           L.max_sweeps, L.tol2, L.KK, L.status);
    });
  }
  R.gemm(Z, 0, 0, k, sP, L.WU, 0, 0, r, static_cast<int64_t>(k) * r, Uout, r, sU, d, r, k);
}

}  // namespace

cudaError_t launch_cl_eig(const float* A, const float* P, float* Wout, float* lam, int d, int batch, int max_sweeps,
                          float tol2, uint32_t* status, cudaStream_t st) {
  if (d > kLK) return cudaErrorInvalidValue;
  cudaError_t e = cl_attributes();
  if (e != cudaSuccess) return e;
  k_cl_svd<<<batch, kLThreads, kk_smem(d), st>>>(A, P, nullptr, Wout, lam, d, d, max_sweeps, tol2, nullptr, status);
  return cudaGetLastError();
}

cudaError_t launch_cl_prep(const void* G, int g_bf16, float* out, int64_t mn, int batch, uint32_t* status,
                           cudaStream_t st) {
  const int64_t gx = (mn + 255) / 256;
  const dim3 grid(static_cast<unsigned>(gx < 256 ? (gx > 0 ? gx : 1) : 256), static_cast<unsigned>(batch));
  if (g_bf16)
    k_cl_prep<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(G), out, mn, status);
  else
    k_cl_prep<float><<<grid, 256, 0, st>>>(static_cast<const float*>(G), out, mn, status);
  return cudaGetLastError();
}

cudaError_t clean_large_refresh(const ClLarge& L, cudaStream_t st, int* launches) {
  cudaError_t e = cl_attributes();
  if (e != cudaSuccess) return e;
  ClRun R{L, st, launches};
  cl_nystrom(R, 0);
  cl_nystrom(R, 1);
  if (L.warm) {
    // Eqns. (14)-(15): O_L = U_Ln^T U_L, O_R = U_R^T U_Rn
    const int m = L.m, n = L.n, r = L.r, k = L.k;
    const int64_t sR = static_cast<int64_t>(r) * r, sK = static_cast<int64_t>(k) * k;
    const int64_t sMA = static_cast<int64_t>(m) * r, sMB = static_cast<int64_t>(r) * n, sUR = static_cast<int64_t>(n) * r;
    float* OL = L.Sm;
    float* OR = L.S;
    R.gemm(L.ULn, 0, 1, r, sMA, L.UL, 0, 0, r, sMA, OL, r, sR, r, r, m);
    R.gemm(L.UR, 0, 1, r, sUR, L.URn, 0, 0, r, sUR, OR, r, sR, r, r, n);
    // M <- O_L M O_R
    R.gemm(OL, 0, 0, r, sR, L.M, 0, 0, r, sR, L.Nm, r, sR, r, r, r);
    R.gemm(L.Nm, 0, 0, r, sR, OR, 0, 0, r, sR, L.Mn, r, sR, r, r, r);
    // M_A <- (I - U_Ln U_Ln^T) M_A O_R
    R.gemm(L.MA, 0, 0, r, sMA, OR, 0, 0, r, sR, L.MAn, r, sMA, m, r, r);
    R.gemm(L.ULn, 0, 1, r, sMA, L.MAn, 0, 0, r, sMA, L.Gram, r, sK, r, r, m);
    R.gemm(L.ULn, 0, 0, r, sMA, L.Gram, 0, 0, r, sK, L.MAn, r, sMA, m, r, r, -1.0f, 1.0f);
    // M_B <- O_L M_B (I - U_Rn U_Rn^T)
    R.gemm(OL, 0, 0, r, sR, L.MB, 0, 0, n, sMB, L.MBn, n, sMB, r, n, r);
    R.gemm(L.MBn, 0, 0, n, sMB, L.URn, 0, 0, r, sUR, L.Rinv, r, sK, r, r, n);
    R.gemm(L.Rinv, 0, 0, r, sK, L.URn, 0, 1, r, sUR, L.MBn, n, sMB, r, n, r, -1.0f, 1.0f);
    R.launch([&] { k_cl_vrot<<<L.batch, 128, 0, st>>>(L.vA, L.vB, OL, OR, L.vAn, L.vBn, r); });
  }
  R.launch([&] {
    const int64_t big = static_cast<int64_t>(L.m > L.n ? L.m : L.n) * L.r;
    k_cl_install<<<R.grid_for(big > static_cast<int64_t>(L.r) * L.n ? big : static_cast<int64_t>(L.r) * L.n), 256, 0,
                   st>>>(L);
  });
  return R.err;
}

cudaError_t clean_large_step(const ClLarge& L, cudaStream_t st, int* launches) {
  ClRun R{L, st, launches};
  const int m = L.m, n = L.n, r = L.r;
  const int64_t mn = static_cast<int64_t>(m) * n, sMA = static_cast<int64_t>(m) * r;
  const int64_t sMB = static_cast<int64_t>(r) * n, sUR = static_cast<int64_t>(n) * r, sR = static_cast<int64_t>(r) * r;
  const int gb = L.g_bf16;
  R.launch([&] {
    if (gb)
      k_cl_prep<__nv_bfloat16><<<R.grid_for(mn), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(L.G), L.Cb, mn,
                                                                L.status);
    else
      k_cl_prep<float><<<R.grid_for(mn), 256, 0, st>>>(static_cast<const float*>(L.G), L.Cb, mn, L.status);
  });
  // G U_R, U_L^T G, S = U_L^T G U_R
  R.gemm(L.G, gb, 0, n, mn, L.UR, 0, 0, r, sUR, L.GU, r, sMA, m, r, n);
  R.gemm(L.UL, 0, 1, r, sMA, L.G, gb, 0, n, mn, L.UG, n, sMB, r, n, m);
  R.gemm(L.UL, 0, 1, r, sMA, L.GU, 0, 0, r, sMA, L.S, r, sR, r, r, m);
  // G_B = U_L^T G - S U_R^T;  C = G - U_L G_B - (G U_R) U_R^T;  G_A = G U_R - U_L S
  R.gemm(L.S, 0, 0, r, sR, L.UR, 0, 1, r, sUR, L.UG, n, sMB, r, n, r, -1.0f, 1.0f);
  R.gemm(L.UL, 0, 0, r, sMA, L.UG, 0, 0, n, sMB, L.Cb, n, mn, m, n, r, -1.0f, 1.0f);
  R.gemm(L.GU, 0, 0, r, sMA, L.UR, 0, 1, r, sUR, L.Cb, n, mn, m, n, r, -1.0f, 1.0f);
  R.gemm(L.UL, 0, 0, r, sMA, L.S, 0, 0, r, sR, L.GU, r, sMA, m, r, r, -1.0f, 1.0f);
  // moments (Table 1) and the normalised blocks
  R.launch([&] { k_cl_sumsq<<<dim3(kClParts, L.batch), 256, 0, st>>>(L.Cb, mn, L.part); });
  R.launch([&] { k_cl_moments<<<L.batch, 256, 0, st>>>(L); });
  R.launch([&] { k_cl_blocks<<<R.grid_for(sMA + sMB), 256, 0, st>>>(L); });
  // G~ = C cden + (U_L N(M, V) + N(M_A, v_A)) U_R^T + U_L N(M_B, v_B)
  R.gemm(L.UL, 0, 0, r, sMA, L.Nm, 0, 0, r, sR, L.GU, r, sMA, m, r, r, 1.0f, 1.0f);
  R.gemm(L.GU, 0, 0, r, sMA, L.UR, 0, 1, r, sUR, L.Cb, n, mn, m, n, r, 1.0f, 0.0f, L.cden);
  R.gemm(L.UL, 0, 0, r, sMA, L.UG, 0, 0, n, sMB, L.Cb, n, mn, m, n, r, 1.0f, 1.0f);
  R.launch([&] {
    if (L.w_bf16)
      k_cl_update<__nv_bfloat16><<<R.grid_for(mn), 256, 0, st>>>(static_cast<__nv_bfloat16*>(L.W), L.Cb, mn, L.decay,
                                                                  L.alr, L.status);
    else
      k_cl_update<float><<<R.grid_for(mn), 256, 0, st>>>(static_cast<float*>(L.W), L.Cb, mn, L.decay, L.alr,
                                                          L.status);
  });
  return R.err;
}

}  // namespace okls

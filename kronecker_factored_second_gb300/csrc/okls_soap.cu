// SOAP step and eigenbasis refresh for matrices with m, n <= 128 (sm_103a).
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching", Appendix C, Algorithm 4 (SOAP), with the KPOP page's section on
// Adam in the Kronecker-factored eigenbasis:
//   G' = Q_L^T G Q_R;  M <- b1 M + (1-b1) G;  M' = Q_L^T M Q_R;
//   V <- b2 V + (1-b2) G' (.) G';  N' = (M'/(1-b1^t)) / (sqrt(V/(1-b2^t)) + eps);
//   N = Q_L N' Q_R^T;  W <- W - decay W - lr N;
//   L <- b2 L + (1-b2) G G^T;  R <- b2 R + (1-b2) G^T G;
//   every f steps: Q_L, Q_R <- eigenvectors of L, R (decreasing eigenvalues,
//   signs aligned with the previous bases).
// One CTA per matrix, fp32 on the CUDA cores: at these sizes a product is
// ~2 M FMAs, and the eigenbasis must be accurate to fp32, not binary16.
// The eigenvectors come from a cyclic Jacobi iteration in shared memory
// (round-robin pairing: d/2 disjoint rotations per round, d-1 rounds per
// sweep), which converges quadratically and keeps the basis orthogonal.
#include <cuda_bf16.h>

#include "okls_internal.h"
#include "okls_kernels.h"
#include "okls_tile.cuh"

namespace okls {

constexpr int kSoapMax = 128;
constexpr int kSoapThreads = 256;
constexpr int kSoapRefThreads = 512;
constexpr int kSoapLd = kSoapMax + 4;                           // padded fp32 pitch (16-byte rows)
constexpr int kSoapBuf = kSoapMax * kSoapLd;                     // floats per staged matrix
constexpr int kSoapStepSmem = 3 * kSoapBuf * 4;                  // three staged matrices
constexpr int kSoapRefreshSmem = 3 * kSoapMax * (kSoapMax + 1) * 4 + 4096;  // A, V, T (+ rotations)

// Copy a rows x cols fp32 matrix (row-major, pitch cols) into shared memory.
__device__ __forceinline__ void soap_stage(float* dst, const float* src, int rows, int cols) {
  for (int e = threadIdx.x; e < rows * cols; e += blockDim.x) dst[(e / cols) * kSoapLd + e % cols] = src[e];
}

// Product of two staged matrices, r x c = op(A) op(B) with K = k; each thread
// forms 4 x 4 outputs and hands each of them to `out(i, j, value)`.
// ta: A is staged k x r (use its transpose); tb: B is staged c x k.
template <class F>
__device__ __forceinline__ void soap_mm4(const float* A, bool ta, const float* B, bool tb, int r, int c, int k,
                                         F&& out) {
  const int tr = (r + 3) / 4, tcn = (c + 3) / 4;
  for (int blk = threadIdx.x; blk < tr * tcn; blk += blockDim.x) {
    const int i0 = (blk / tcn) * 4, j0 = (blk % tcn) * 4;
    float acc[4][4] = {};
    for (int q = 0; q < k; ++q) {
      float av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = ta ? A[q * kSoapLd + i0 + u] : A[(i0 + u) * kSoapLd + q];
        bv[u] = tb ? B[(j0 + u) * kSoapLd + q] : B[q * kSoapLd + j0 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        if (i0 + u < r && j0 + v < c) out(i0 + u, j0 + v, acc[u][v]);
  }
}

template <typename WT>
__device__ __forceinline__ float w_load(const WT* p);
template <>
__device__ __forceinline__ float w_load<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float w_load<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void w_store(float* p, float v) { *p = v; }
__device__ __forceinline__ void w_store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// One matrix per CTA.  Shared memory holds three staged matrices: G (later
// N'), a basis (Q_L or Q_R, staged for each product) and one intermediate.
// Out-of-range rows and columns of the staged tiles are zero, so the 4 x 4
// tiles never read garbage.
template <typename WT, typename GT>
__global__ void __launch_bounds__(kSoapThreads) k_soap_step(SoapArgs A) {
  extern __shared__ float sm[];
  // this grid raises the status word itself: one read per block keeps the
  // early exit uniform across the block's threads
  if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(A.status) != 0u)) return;
  const int b = blockIdx.x;
  const int m = A.m, n = A.n;
  const int64_t mn = static_cast<int64_t>(m) * n;
  float* Gs = sm;                 // G, then N'
  float* Qs = sm + kSoapBuf;      // Q_L or Q_R
  float* Ts = sm + 2 * kSoapBuf;  // left halves of the two-sided products
  const GT* G = static_cast<const GT*>(A.G) + b * mn;
  WT* W = static_cast<WT*>(A.W) + b * mn;
  float* M = A.M + b * mn;
  float* V = A.V + b * mn;
  float* L = A.L + static_cast<int64_t>(b) * m * m;
  float* R = A.R + static_cast<int64_t>(b) * n * n;
  const float* QL = A.QL + static_cast<int64_t>(b) * m * m;
  const float* QR = A.QR + static_cast<int64_t>(b) * n * n;
  bool bad = false;

  for (int e = threadIdx.x; e < 3 * kSoapBuf; e += blockDim.x) sm[e] = 0.0f;
  __syncthreads();
  for (int e = threadIdx.x; e < mn; e += blockDim.x) {
    const float g = w_load<GT>(G + e);
    bad |= !isfinite(g);
    Gs[(e / n) * kSoapLd + e % n] = g;
  }
  soap_stage(Qs, QL, m, m);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) atomicOr(A.status, kStNonfiniteInput);
    return;
  }
  // G' = Q_L^T G Q_R, straight into V <- b2 V + (1-b2) G'^2
  soap_mm4(Qs, true, Gs, false, m, n, m, [&](int i, int j, float v) { Ts[i * kSoapLd + j] = v; });
  __syncthreads();
  soap_stage(Qs, QR, n, n);
  __syncthreads();
  soap_mm4(Ts, false, Qs, false, m, n, n, [&](int i, int j, float v) {
    float& x = V[static_cast<int64_t>(i) * n + j];
    x = fmaf(A.beta2, x, (1.0f - A.beta2) * v * v);
  });
  // M <- b1 M + (1-b1) G; L <- b2 L + (1-b2) G G^T; R <- b2 R + (1-b2) G^T G
  for (int e = threadIdx.x; e < mn; e += blockDim.x)
    M[e] = fmaf(A.beta1, M[e], (1.0f - A.beta1) * Gs[(e / n) * kSoapLd + e % n]);
  soap_mm4(Gs, false, Gs, true, m, m, n, [&](int i, int j, float v) {
    float& x = L[static_cast<int64_t>(i) * m + j];
    x = fmaf(A.beta2, x, (1.0f - A.beta2) * v);
  });
  soap_mm4(Gs, true, Gs, false, n, n, m, [&](int i, int j, float v) {
    float& x = R[static_cast<int64_t>(i) * n + j];
    x = fmaf(A.beta2, x, (1.0f - A.beta2) * v);
  });
  __syncthreads();
  // M' = Q_L^T M Q_R, then N' = (M'/(1-b1^t)) / (sqrt(V/(1-b2^t)) + eps) into Gs
  for (int e = threadIdx.x; e < mn; e += blockDim.x) Gs[(e / n) * kSoapLd + e % n] = M[e];
  soap_stage(Qs, QL, m, m);
  __syncthreads();
  soap_mm4(Qs, true, Gs, false, m, n, m, [&](int i, int j, float v) { Ts[i * kSoapLd + j] = v; });
  __syncthreads();
  soap_stage(Qs, QR, n, n);
  __syncthreads();
  soap_mm4(Ts, false, Qs, false, m, n, n, [&](int i, int j, float v) {
    const float vv = V[static_cast<int64_t>(i) * n + j];
    Gs[i * kSoapLd + j] = (v * A.bc1) / (sqrtf(vv * A.bc2) + A.eps);
  });
  __syncthreads();
  // N = Q_L N' Q_R^T and the update
  soap_stage(Qs, QL, m, m);
  __syncthreads();
  soap_mm4(Qs, false, Gs, false, m, n, m, [&](int i, int j, float v) { Ts[i * kSoapLd + j] = v; });
  __syncthreads();
  soap_stage(Qs, QR, n, n);
  __syncthreads();
  soap_mm4(Ts, false, Qs, true, m, n, n, [&](int i, int j, float v) {
    WT* w = W + static_cast<int64_t>(i) * n + j;
    const float nw = fmaf(-A.lr, v, A.decay * w_load<WT>(w));
    bad |= !isfinite(nw);
    w_store(w, nw);
  });
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(A.status, kStNonfiniteUpdate);
}

// ------------------------------------------------------------------ refresh
// Round-robin pairing of d' = d rounded up to even indices, round r:
// position 0 stays, the others rotate; pair (pos k, pos d'-1-k).
__device__ __forceinline__ int rr_index(int pos, int r, int dp) {
  if (pos == 0) return 0;
  return 1 + (pos - 1 + r) % (dp - 1);
}

__global__ void __launch_bounds__(kSoapRefThreads) k_soap_refresh(SoapRefreshArgs A) {
  extern __shared__ float sm[];
  if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(A.status) != 0u)) return;
  const int fi = blockIdx.x < A.count ? 0 : 1;
  const int b = fi == 0 ? blockIdx.x : blockIdx.x - A.count;
  const int d = fi == 0 ? A.d0 : A.d1;
  const float* S = (fi == 0 ? A.S0 : A.S1) + static_cast<int64_t>(b) * d * d;
  float* Q = (fi == 0 ? A.Q0 : A.Q1) + static_cast<int64_t>(b) * d * d;
  const int ld = kSoapMax + 1;
  float* As = sm;                    // the matrix being diagonalised
  float* Vs = sm + kSoapMax * ld;    // accumulated rotations (eigenvectors in columns)
  float* Ts = Vs + kSoapMax * ld;    // the polished previous basis
  float* cs = Ts + kSoapMax * ld;    // per pair: c, s
  int* pr = reinterpret_cast<int*>(cs + kSoapMax);  // per pair: p, q
  __shared__ float red[kSoapRefThreads / 32];
  __shared__ float off_sum, diag_sum;
  const int dp = d + (d & 1);
  const int np = dp / 2;
  // Warm start from the previous basis Q (the argument of Eigenvectors(L, Q_L)):
  // Q^ = Q (3 I - Q^T Q) / 2 (one polar step: keeps the basis orthogonal to
  // the fp32 floor however many refreshes it has been through), then the
  // iteration starts from A = Q^^T S Q^ and V = Q^.  With Q = I (the first
  // refresh) every step is exact and this is the plain Jacobi start.
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) Vs[(e / d) * ld + e % d] = Q[e];
  __syncthreads();
  tile_mm4(Vs, ld, true, Vs, ld, false, d, d, d,
           [&](int i, int j, float v) { As[i * ld + j] = (i == j ? 1.5f : 0.0f) - 0.5f * v; });
  __syncthreads();
  tile_mm4(Vs, ld, false, As, ld, false, d, d, d, [&](int i, int j, float v) { Ts[i * ld + j] = v; });
  __syncthreads();
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) {
    const int i = e / d, j = e % d;
    As[i * ld + j] = 0.5f * (S[i * d + j] + S[j * d + i]);
  }
  __syncthreads();
  tile_mm4(As, ld, false, Ts, ld, false, d, d, d, [&](int i, int j, float v) { Vs[i * ld + j] = v; });  // S Q^
  __syncthreads();
  tile_mm4(Ts, ld, true, Vs, ld, false, d, d, d, [&](int i, int j, float v) { As[i * ld + j] = v; });  // Q^T S Q^
  __syncthreads();
  for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
    const int i = e / dp, j = e % dp;
    if (i < d && j < d) {
      if (i < j) {
        const float v = 0.5f * (As[i * ld + j] + As[j * ld + i]);
        As[i * ld + j] = v;
        As[j * ld + i] = v;
      }
      Vs[i * ld + j] = Ts[i * ld + j];
    } else {
      As[i * ld + j] = 0.0f;  // the padding index of an odd d
      Vs[i * ld + j] = i == j ? 1.0f : 0.0f;
    }
  }
  __syncthreads();
  for (int sweep = 0; sweep < A.max_sweeps; ++sweep) {
    // convergence: off-diagonal mass against the diagonal's
    float off = 0.0f, dg = 0.0f;
    for (int e = threadIdx.x; e < dp * dp; e += blockDim.x) {
      const int i = e / dp, j = e % dp;
      const float v = As[i * ld + j];
      if (i == j)
        dg = fmaf(v, v, dg);
      else
        off = fmaf(v, v, off);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      off += __shfl_xor_sync(0xffffffffu, off, o);
      dg += __shfl_xor_sync(0xffffffffu, dg, o);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = off;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < kSoapRefThreads / 32; ++w) t += red[w];
      off_sum = t;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dg;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < kSoapRefThreads / 32; ++w) t += red[w];
      diag_sum = t;
    }
    __syncthreads();
    if (!(off_sum > A.tol2 * diag_sum)) break;
    for (int r = 0; r < dp - 1; ++r) {
      // 1. rotations of the d'/2 disjoint pairs of this round
      for (int k = threadIdx.x; k < np; k += blockDim.x) {
        int p = rr_index(k, r, dp), q = rr_index(dp - 1 - k, r, dp);
        if (p > q) {
          const int x = p;
          p = q;
          q = x;
        }
        const float apq = As[p * ld + q];
        float c = 1.0f, s = 0.0f;
        if (apq != 0.0f) {
          const float theta = (As[q * ld + q] - As[p * ld + p]) / (2.0f * apq);
          const float t = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(fmaf(theta, theta, 1.0f)));
          c = rsqrtf(fmaf(t, t, 1.0f));
          s = t * c;
        }
        cs[2 * k] = c;
        cs[2 * k + 1] = s;
        pr[2 * k] = p;
        pr[2 * k + 1] = q;
      }
      __syncthreads();
      // threads: lane j = tid % 128 walks a row or column, group tid / 128 a
      // quarter of the pairs
      const int j = threadIdx.x & (kSoapMax - 1);
      const int g0 = threadIdx.x >> 7;
      constexpr int kGroups = kSoapRefThreads / kSoapMax;
      // 2. rows p, q of A (A <- J^T A)
      if (j < dp) {
        for (int k = g0; k < np; k += kGroups) {
          const int p = pr[2 * k], q = pr[2 * k + 1];
          const float c = cs[2 * k], s = cs[2 * k + 1];
          const float ap = As[p * ld + j], aq = As[q * ld + j];
          As[p * ld + j] = c * ap - s * aq;
          As[q * ld + j] = s * ap + c * aq;
        }
      }
      __syncthreads();
      // 3. columns p, q of A (A <- A J) and of V (V <- V J); j is the row here
      if (j < dp) {
        for (int k = g0; k < np; k += kGroups) {
          const int p = pr[2 * k], q = pr[2 * k + 1];
          const float c = cs[2 * k], s = cs[2 * k + 1];
          const float ap = As[j * ld + p], aq = As[j * ld + q];
          As[j * ld + p] = c * ap - s * aq;
          As[j * ld + q] = s * ap + c * aq;
          const float vp = Vs[j * ld + p], vq = Vs[j * ld + q];
          Vs[j * ld + p] = c * vp - s * vq;
          Vs[j * ld + q] = s * vp + c * vq;
        }
      }
      __syncthreads();
    }
  }
  // 4. eigenvalues in decreasing order (ties by index), signs aligned with
  //    the previous basis; column j of Q is the eigenvector of rank j
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float lj = As[j * ld + j];
    int rank = 0;
    for (int i = 0; i < d; ++i) {
      const float li = As[i * ld + i];
      rank += (li > lj) || (li == lj && i < j);
    }
    float dot = 0.0f;
    for (int i = 0; i < d; ++i) dot = fmaf(Vs[i * ld + j], Q[i * d + rank], dot);
    cs[j] = dot < 0.0f ? -1.0f : 1.0f;
    pr[2 * kSoapMax / 2 + j] = rank;  // second half of the pair table
  }
  __syncthreads();
  const int* rank_of = pr + kSoapMax;
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) {
    const int i = e / d, j = e % d;
    Q[i * d + rank_of[j]] = cs[j] * Vs[i * ld + j];
  }
}

// M = V = 0, L = R = 0, Q_L = Q_R = I (the bases before the first refresh)
__global__ void k_soap_reset(float* M, float* V, float* L, float* R, float* QL, float* QR, int m, int n) {
  const int b = blockIdx.y;
  const int64_t mn = static_cast<int64_t>(m) * n;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    M[b * mn + e] = 0.0f;
    V[b * mn + e] = 0.0f;
  }
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < static_cast<int64_t>(m) * m;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    L[b * static_cast<int64_t>(m) * m + e] = 0.0f;
    QL[b * static_cast<int64_t>(m) * m + e] = (e / m == e % m) ? 1.0f : 0.0f;
  }
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < static_cast<int64_t>(n) * n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    R[b * static_cast<int64_t>(n) * n + e] = 0.0f;
    QR[b * static_cast<int64_t>(n) * n + e] = (e / n == e % n) ? 1.0f : 0.0f;
  }
}

cudaError_t launch_soap_reset(float* M, float* V, float* L, float* R, float* QL, float* QR, int batch, int m, int n,
                              cudaStream_t st) {
  k_soap_reset<<<dim3(8, batch), 256, 0, st>>>(M, V, L, R, QL, QR, m, n);
  return cudaGetLastError();
}

// opt in to the large dynamic shared memory of both kernels, once per device
static cudaError_t soap_attributes() {
  static PerDevice pd;
  return once_per_device(pd, [](int) {
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(k_soap_step<float, float>, at, kSoapStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_soap_step<float, __nv_bfloat16>, at, kSoapStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_soap_step<__nv_bfloat16, float>, at, kSoapStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_soap_step<__nv_bfloat16, __nv_bfloat16>, at, kSoapStepSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_soap_refresh, at, kSoapRefreshSmem);
    return e;
  });
}

cudaError_t launch_soap_step(const SoapArgs& A, cudaStream_t st) {
  cudaError_t e = soap_attributes();
  if (e != cudaSuccess) return e;
  if (A.w_bf16 && A.g_bf16)
    k_soap_step<__nv_bfloat16, __nv_bfloat16><<<A.batch, kSoapThreads, kSoapStepSmem, st>>>(A);
  else if (A.w_bf16)
    k_soap_step<__nv_bfloat16, float><<<A.batch, kSoapThreads, kSoapStepSmem, st>>>(A);
  else if (A.g_bf16)
    k_soap_step<float, __nv_bfloat16><<<A.batch, kSoapThreads, kSoapStepSmem, st>>>(A);
  else
    k_soap_step<float, float><<<A.batch, kSoapThreads, kSoapStepSmem, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_soap_refresh(const SoapRefreshArgs& A, cudaStream_t st) {
  cudaError_t e = soap_attributes();
  if (e != cudaSuccess) return e;
  k_soap_refresh<<<2 * A.count, kSoapRefThreads, kSoapRefreshSmem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace okls

// Batched symmetric eigensolver for k x k matrices, 128 < k <= kClMaxK
// (sm_103a): cyclic Jacobi with the rotations of each sweep logged and
// applied to the eigenvector matrix by a separate, wide kernel.
//
// Used by the SOAP refresh (Clean page, Appendix C, Algorithm 4:
// Eigenvectors(L, Q_L)) and by Clean's thin SVD of the sketch (Clean page,
// Appendix A, Algorithm 3: the eigen-decomposition of Z^T Z).
//
// Per sweep, two launches:
//   k_eig_sweep  one CTA per matrix.  The matrix A sits as a packed upper
//                triangle in shared memory up to kEigPackMaxK, and as a full
//                symmetric dp x dp matrix in an L2-resident scratch slice past
//                it (every access of a round is then a contiguous run of a
//                row).  The sweep's stopping rule is checked first; then each
//                of the dp - 1 rounds of the round-robin ordering computes its
//                dp / 2 disjoint rotations (threshold Jacobi: a pair whose
//                off-diagonal entry is already below tol2 / k of its diagonal
//                is left alone), writes them to the sweep's log and applies
//                J^T A J as one pass over the 2 x 2 blocks of every two pairs.
//   k_eig_apply  V <- V J for every logged rotation, on rows of V: rows are
//                independent under right multiplication, so each CTA keeps a
//                band of rows in shared memory and runs all rounds on it, and
//                the work spreads over batch x k / kApplyRows CTAs instead of
//                batch.
// k_eig_finish orders the eigenpairs by decreasing eigenvalue, chooses each
// column's sign against the previous basis and writes the requested columns.
//
// The full-matrix pass keeps A bit-exactly symmetric: the 2 x 2 block of the
// unordered pair {x, y}, x <= y, is always formed as (J_x^T B) J_y from the
// block B with x's rows, and the item that owns the transposed block writes
// the transpose of the same result.
#include <algorithm>

#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

namespace {

constexpr int kEigPackMaxK = 330;  // packed triangle in shared memory up to here
constexpr int kEigThreads = 1024;
constexpr int kApplyRows = 32;
constexpr int kApplyThreads = 256;
constexpr int kFinishThreads = 512;
constexpr int kEigHead = 4 * kClMaxK;  // floats: rotations (2 per pair), pairs (2 per pair)

struct EigSlice {
  float* A;      // dp x dp (full) or dp (dp + 1) / 2 (packed)
  float* V;      // k x k, row-major
  float2* log;   // (dp - 1) x (dp / 2) rotations (c, s) of the current sweep
  int* flags;    // [0] still active, [1] rotated in the current sweep
};

__host__ __device__ inline int64_t round4(int64_t x) { return (x + 3) & ~int64_t(3); }

__host__ __device__ inline int64_t slice_floats(int k) {
  const int64_t dp = k + (k & 1);
  return round4(dp * dp) + round4(static_cast<int64_t>(k) * k) + round4((dp - 1) * dp) + 4;
}

__device__ __forceinline__ EigSlice eig_slice(float* scratch, int k, int b) {
  const int64_t dp = k + (k & 1);
  float* base = scratch + static_cast<int64_t>(b) * slice_floats(k);
  EigSlice s;
  s.A = base;
  s.V = base + round4(dp * dp);
  s.log = reinterpret_cast<float2*>(s.V + round4(static_cast<int64_t>(k) * k));
  s.flags = reinterpret_cast<int*>(reinterpret_cast<float*>(s.log) + round4((dp - 1) * dp));
  return s;
}

// which side and which matrix of it a block works on; sub = block within the matrix
struct Where {
  const EigSide* side;
  int b, sub;
};

__device__ __forceinline__ Where locate(const EigPlan& P, int blocks_per_matrix0, int blocks_per_matrix1) {
  const int x = blockIdx.x;
  const int n0 = P.side[0].count * blocks_per_matrix0;
  if (x < n0) return {&P.side[0], x / blocks_per_matrix0, x % blocks_per_matrix0};
  const int y = x - n0;
  return {&P.side[1], y / blocks_per_matrix1, y % blocks_per_matrix1};
}

__device__ __forceinline__ bool eig_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

__device__ __forceinline__ float eig_block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
  return s;
}

__device__ __forceinline__ int pk(int i, int j, int dp) {  // i <= j
  return i * dp - (i * (i - 1)) / 2 + (j - i);
}

// the pair of position q in round rd of the round-robin ordering, p < q
__device__ __forceinline__ void round_pair(int q, int rd, int dp, int& pp, int& qq) {
  auto idx = [&](int pos) { return pos == 0 ? 0 : 1 + (pos - 1 + rd) % (dp - 1); };
  pp = idx(q);
  qq = idx(dp - 1 - q);
  if (pp > qq) {
    const int x = pp;
    pp = qq;
    qq = x;
  }
}

// n = (J1^T X) J2 with J = [[c, s], [-s, c]]
struct Blk {
  float a11, a12, a21, a22;
};
__device__ __forceinline__ Blk rot2(const Blk x, float c1, float s1, float c2, float s2) {
  const float r11 = fmaf(c1, x.a11, -(s1 * x.a21)), r12 = fmaf(c1, x.a12, -(s1 * x.a22));
  const float r21 = fmaf(s1, x.a11, c1 * x.a21), r22 = fmaf(s1, x.a12, c1 * x.a22);
  Blk n;
  n.a11 = fmaf(c2, r11, -(s2 * r12));
  n.a12 = fmaf(s2, r11, c2 * r12);
  n.a21 = fmaf(c2, r21, -(s2 * r22));
  n.a22 = fmaf(s2, r21, c2 * r22);
  return n;
}

// the rotation zeroing a_pq (left alone below the threshold)
__device__ __forceinline__ float2 jacobi_cs(float app, float aqq, float apq, float skip2) {
  float c = 1.0f, sn = 0.0f;
  if (apq * apq > skip2 * fabsf(app * aqq)) {
    const float th = (aqq - app) / (2.0f * apq);
    const float t = copysignf(1.0f, th) / (fabsf(th) + sqrtf(fmaf(th, th, 1.0f)));
    c = rsqrtf(fmaf(t, t, 1.0f));
    sn = t * c;
  }
  return make_float2(c, sn);
}

}  // namespace

// One sweep of cyclic Jacobi on one matrix per CTA.  kFull: A lives as a full
// dp x dp matrix in the scratch slice; else as a packed triangle in shared
// memory, loaded from / stored to the slice around the sweep.
template <bool kFull>
__device__ void sweep_body(const EigPlan& P, const EigSide& S, int b, int sweep, float* sm) {
  __shared__ float red[kEigThreads / 32];
  const int k = S.k;
  const int dp = k + (k & 1), np = dp / 2;
  const EigSlice sl = eig_slice(S.scratch, k, b);
  // a converged matrix stays converged: later sweeps do nothing
  if (sweep > 0 && sl.flags[0] == 0) {
    if (threadIdx.x == 0) sl.flags[1] = 0;
    return;
  }
  float* cs = sm;                                   // 2 per pair
  int* pr = reinterpret_cast<int*>(sm + 2 * kClMaxK);  // 2 per pair
  float* A = kFull ? sl.A : sm + kEigHead;
  const int tid = threadIdx.x, nth = blockDim.x;
  if (sweep == 0) {
    // the symmetric part of the input (bit-exactly symmetric), padded by a
    // zero row and column when k is odd
    const float* G = S.A + static_cast<int64_t>(b) * k * k;
    for (int j = tid; j < dp; j += nth)
      for (int i = 0; i <= j; ++i) {
        const float v = (i < k && j < k) ? 0.5f * (G[i * k + j] + G[j * k + i]) : 0.0f;
        if (kFull) {
          A[static_cast<int64_t>(i) * dp + j] = v;
          A[static_cast<int64_t>(j) * dp + i] = v;
        } else {
          A[pk(i, j, dp)] = v;
        }
      }
  } else if (!kFull) {
    const int npk = dp * (dp + 1) / 2;
    for (int e = tid; e < npk; e += nth) A[e] = sl.A[e];
  }
  __syncthreads();
  float off = 0.0f, dg = 0.0f;
  for (int j = tid; j < dp; j += nth)
    for (int i = 0; i <= j; ++i) {
      const float v = kFull ? A[static_cast<int64_t>(i) * dp + j] : A[pk(i, j, dp)];
      if (i == j)
        dg = fmaf(v, v, dg);
      else
        off = fmaf(2.0f * v, v, off);
    }
  const float offs = eig_block_sum(off, red);
  const float dgs = eig_block_sum(dg, red);
  const bool more = offs > P.tol2 * dgs;
  if (tid == 0) {
    sl.flags[0] = more ? 1 : 0;
    sl.flags[1] = more ? 1 : 0;
  }
  if (more) {
    const float skip2 = P.tol2 / static_cast<float>(k);
    for (int rd = 0; rd < dp - 1; ++rd) {
      for (int q = tid; q < np; q += nth) {
        int pp, qq;
        round_pair(q, rd, dp, pp, qq);
        float app, aqq, apq;
        if (kFull) {
          app = A[static_cast<int64_t>(pp) * dp + pp];
          aqq = A[static_cast<int64_t>(qq) * dp + qq];
          apq = A[static_cast<int64_t>(pp) * dp + qq];
        } else {
          app = A[pk(pp, pp, dp)];
          aqq = A[pk(qq, qq, dp)];
          apq = A[pk(pp, qq, dp)];
        }
        const float2 r = jacobi_cs(app, aqq, apq, skip2);
        cs[2 * q] = r.x;
        cs[2 * q + 1] = r.y;
        pr[2 * q] = pp;
        pr[2 * q + 1] = qq;
        sl.log[static_cast<int64_t>(rd) * np + q] = r;
      }
      __syncthreads();
      if (kFull) {
        // every ordered pair of pairs (x, y): rows {p_x, q_x}, columns {p_y, q_y}
        const int total = np * np;
        int x = tid / np, y = tid - (tid / np) * np;
        const int dx = nth / np, dy = nth - dx * np;
        for (int e = tid; e < total; e += nth) {
          const float c1 = cs[2 * x], s1 = cs[2 * x + 1], c2 = cs[2 * y], s2 = cs[2 * y + 1];
          if (s1 != 0.0f || s2 != 0.0f) {
            const int p1 = pr[2 * x], q1 = pr[2 * x + 1], p2 = pr[2 * y], q2 = pr[2 * y + 1];
            float* r1 = A + static_cast<int64_t>(p1) * dp;
            float* r2 = A + static_cast<int64_t>(q1) * dp;
            const Blk C{r1[p2], r1[q2], r2[p2], r2[q2]};
            if (x == y) {
              const Blk n = rot2(C, c1, s1, c1, s1);
              r1[p1] = n.a11;
              r1[q1] = n.a12;
              r2[p1] = n.a12;
              r2[q1] = n.a22;
            } else if (x < y) {
              const Blk n = rot2(C, c1, s1, c2, s2);
              r1[p2] = n.a11;
              r1[q2] = n.a12;
              r2[p2] = n.a21;
              r2[q2] = n.a22;
            } else {
              // the block of {y, x} is C^T; write the transpose of its result
              const Blk n = rot2(Blk{C.a11, C.a21, C.a12, C.a22}, c2, s2, c1, s1);
              r1[p2] = n.a11;
              r1[q2] = n.a21;
              r2[p2] = n.a12;
              r2[q2] = n.a22;
            }
          }
          x += dx;
          y += dy;
          if (y >= np) {
            y -= np;
            ++x;
          }
        }
      } else {
        // the upper blocks (u <= v) of the packed triangle
        for (int e = tid; e < np * np; e += nth) {
          const int u = e / np, v = e - (e / np) * np;
          if (u > v) continue;
          const float c1 = cs[2 * u], s1 = cs[2 * u + 1], c2 = cs[2 * v], s2 = cs[2 * v + 1];
          if (s1 == 0.0f && s2 == 0.0f) continue;
          const int p1 = pr[2 * u], q1 = pr[2 * u + 1], p2 = pr[2 * v], q2 = pr[2 * v + 1];
          auto get = [&](int i, int j) { return i <= j ? A[pk(i, j, dp)] : A[pk(j, i, dp)]; };
          auto set = [&](int i, int j, float val) {
            if (i <= j)
              A[pk(i, j, dp)] = val;
            else
              A[pk(j, i, dp)] = val;
          };
          const Blk n = rot2(Blk{get(p1, p2), get(p1, q2), get(q1, p2), get(q1, q2)}, c1, s1, c2, s2);
          if (u == v) {
            set(p1, p1, n.a11);
            set(p1, q1, n.a12);
            set(q1, q1, n.a22);
          } else {
            set(p1, p2, n.a11);
            set(p1, q2, n.a12);
            set(q1, p2, n.a21);
            set(q1, q2, n.a22);
          }
        }
      }
      __syncthreads();
    }
  }
  // the packed triangle goes back to the slice for the next sweep and the
  // finishing kernel (at sweep 0 also when nothing rotated: it was built here)
  if (!kFull && (more || sweep == 0)) {
    const int npk = dp * (dp + 1) / 2;
    for (int e = tid; e < npk; e += nth) sl.A[e] = A[e];
  }
}

__global__ void __launch_bounds__(kEigThreads) k_eig_sweep(const __grid_constant__ EigPlan P, int sweep) {
  extern __shared__ float sm[];
  if (eig_flagged(P.status)) return;
  const Where w = locate(P, 1, 1);
  if (w.side->k > kEigPackMaxK)
    sweep_body<true>(P, *w.side, w.b, sweep, sm);
  else
    sweep_body<false>(P, *w.side, w.b, sweep, sm);
}

// V <- V J for the rotations logged by sweep `sweep`, on a band of
// kApplyRows rows of V per CTA (V = I before sweep 0).
__global__ void __launch_bounds__(kApplyThreads) k_eig_apply(const __grid_constant__ EigPlan P, int sweep,
                                                            int bands0, int bands1) {
  extern __shared__ float vs[];
  if (eig_flagged(P.status)) return;
  const Where w = locate(P, bands0, bands1);
  const int k = w.side->k;
  const int dp = k + (k & 1), np = dp / 2;
  const EigSlice sl = eig_slice(w.side->scratch, k, w.b);
  const bool ran = sl.flags[1] != 0;
  if (sweep > 0 && !ran) return;
  const int l0 = w.sub * kApplyRows;
  const int rows = min(kApplyRows, k - l0);
  const int tid = threadIdx.x, nth = blockDim.x;
  for (int e = tid; e < kApplyRows * dp; e += nth) {
    const int r = e / dp, j = e - (e / dp) * dp;
    float v = 0.0f;
    if (r < rows && j < k) v = sweep == 0 ? (l0 + r == j ? 1.0f : 0.0f) : sl.V[static_cast<int64_t>(l0 + r) * k + j];
    vs[e] = v;
  }
  __syncthreads();
  if (ran) {
    // each thread owns pairs q = tid, tid + nth, ...; the next round's
    // rotations are fetched while the current round runs
    const int nq = (np + nth - 1) / nth;  // at most 2 for k <= kClMaxK
    float2 cur[2], nxt[2];
    for (int i = 0; i < 2; ++i) {
      const int q = tid + i * nth;
      cur[i] = (i < nq && q < np) ? sl.log[q] : make_float2(1.0f, 0.0f);
    }
    for (int rd = 0; rd < dp - 1; ++rd) {
      for (int i = 0; i < 2; ++i) {
        const int q = tid + i * nth;
        nxt[i] = (rd + 1 < dp - 1 && i < nq && q < np) ? sl.log[static_cast<int64_t>(rd + 1) * np + q]
                                                       : make_float2(1.0f, 0.0f);
      }
      for (int i = 0; i < 2; ++i) {
        const int q = tid + i * nth;
        const float c = cur[i].x, sn = cur[i].y;
        if (i < nq && q < np && sn != 0.0f) {
          int pp, qq;
          round_pair(q, rd, dp, pp, qq);
          for (int r = 0; r < rows; ++r) {
            float* row = vs + r * dp;
            const float vp = row[pp], vq = row[qq];
            row[pp] = fmaf(c, vp, -(sn * vq));
            row[qq] = fmaf(sn, vp, c * vq);
          }
        }
      }
      __syncthreads();
      cur[0] = nxt[0];
      cur[1] = nxt[1];
    }
  }
  for (int e = tid; e < rows * k; e += nth) {
    const int r = e / k, j = e - (e / k) * k;
    sl.V[static_cast<int64_t>(l0 + r) * k + j] = vs[r * dp + j];
  }
}

// Eigenpairs ordered by decreasing eigenvalue (ties by index); column c of W
// is s_c v_j / sigma_j (nu given: Clean's thin SVD, sigma_j^2 the eigenvalue)
// or s_c v_j (nu null) for the pair j of rank c < r, s_c = +-1 making its
// product with column c of P non-negative (P null: +1); lam_c is the
// eigenvalue, less nu and clamped at zero when nu is given.
__global__ void __launch_bounds__(kFinishThreads) k_eig_finish(const __grid_constant__ EigPlan P) {
  __shared__ float dg[kClMaxK];
  __shared__ int rk[kClMaxK];
  if (eig_flagged(P.status)) return;
  const Where w = locate(P, 1, 1);
  const EigSide& S = *w.side;
  const int b = w.b, k = S.k, r = S.r;
  const int dp = k + (k & 1);
  const EigSlice sl = eig_slice(S.scratch, k, b);
  const bool full = k > kEigPackMaxK;
  const int tid = threadIdx.x, nth = blockDim.x;
  for (int j = tid; j < k; j += nth) dg[j] = full ? sl.A[static_cast<int64_t>(j) * dp + j] : sl.A[pk(j, j, dp)];
  __syncthreads();
  for (int j = tid; j < k; j += nth) {
    const float lj = dg[j];
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += (dg[i] > lj) || (dg[i] == lj && i < j);
    rk[j] = rank;
  }
  __syncthreads();
  const bool unit = S.nu == nullptr;
  const float nub = unit ? 0.0f : S.nu[b];
  float* W = S.W + static_cast<int64_t>(b) * k * r;
  const float* Pb = S.P ? S.P + static_cast<int64_t>(b) * k * r : nullptr;
  for (int j = tid; j < k; j += nth) {
    const int c = rk[j];
    if (c >= r) continue;
    const float s2 = dg[j];
    const float inv = unit ? 1.0f : (s2 > 0.0f ? rsqrtf(s2) : 0.0f);
    float sg = 1.0f;
    if (Pb) {
      float dot = 0.0f;
      for (int l = 0; l < k; ++l) dot = fmaf(sl.V[static_cast<int64_t>(l) * k + j], Pb[static_cast<int64_t>(l) * r + c], dot);
      sg = dot < 0.0f ? -1.0f : 1.0f;
    }
    for (int l = 0; l < k; ++l) W[static_cast<int64_t>(l) * r + c] = sg * inv * sl.V[static_cast<int64_t>(l) * k + j];
    if (S.lam) S.lam[static_cast<int64_t>(b) * r + c] = unit ? s2 : fmaxf(0.0f, s2 - nub);
  }
}

size_t eig_scratch_floats(int k) { return static_cast<size_t>(slice_floats(k)); }

namespace {

int sweep_smem(int k) {
  const int dp = k + (k & 1);
  return (kEigHead + (k <= kEigPackMaxK ? dp * (dp + 1) / 2 : 0)) * 4;
}

cudaError_t eig_attributes() {
  static int attr_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || attr_dev == dev) return e;
  const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
  e = cudaFuncSetAttribute(k_eig_sweep, at, sweep_smem(kEigPackMaxK));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_eig_apply, at, kApplyRows * (kClMaxK + 1) * 4);
  if (e == cudaSuccess) attr_dev = dev;
  return e;
}

}  // namespace

cudaError_t launch_eig_rounds(const EigPlan& P, cudaStream_t st, int* launches) {
  for (int i = 0; i < 2; ++i) {
    const EigSide& S = P.side[i];
    if (S.count < 0 || (S.count > 0 && (S.k <= 128 || S.k > kClMaxK || S.r < 1 || S.r > S.k)))
      return cudaErrorInvalidValue;
  }
  if (P.max_sweeps < 1) return cudaErrorInvalidValue;
  const int nb = P.side[0].count + P.side[1].count;
  if (nb == 0) return cudaSuccess;
  cudaError_t e = eig_attributes();
  if (e != cudaSuccess) return e;
  int smem = 0, dpmax = 0, bands[2] = {1, 1}, napply = 0;
  for (int i = 0; i < 2; ++i) {
    const EigSide& S = P.side[i];
    if (S.count == 0) continue;
    smem = std::max(smem, sweep_smem(S.k));
    dpmax = std::max(dpmax, S.k + (S.k & 1));
    bands[i] = (S.k + kApplyRows - 1) / kApplyRows;
    napply += S.count * bands[i];
  }
  const int apply_smem = kApplyRows * dpmax * 4;
  for (int s = 0; s < P.max_sweeps; ++s) {
    k_eig_sweep<<<nb, kEigThreads, smem, st>>>(P, s);
    k_eig_apply<<<napply, kApplyThreads, apply_smem, st>>>(P, s, bands[0], bands[1]);
  }
  k_eig_finish<<<nb, kFinishThreads, 0, st>>>(P);
  if (launches) *launches += 2 * P.max_sweeps + 1;
  return cudaGetLastError();
}

}  // namespace okls

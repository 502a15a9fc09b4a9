// Blocked Jacobi eigensolver for the SOAP refresh past kClMaxK (sm_103a).
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching", Appendix C, Algorithm 4 (SOAP): Eigenvectors(L, Q_L) -- the
// eigenvectors of the factor, ordered by decreasing eigenvalue, each column's
// sign matched to the previous basis.  The caller forms A = Q^^T F Q^ in the
// polar-corrected previous basis Q^; this file diagonalises A and writes
// Q^ W, reordered and sign-aligned, over the previous basis.
//
// The method: two-sided block Jacobi.  A (padded to kp, a multiple of 64, by
// zero rows and columns that no rotation ever touches) is split into
// nb = kp / 32 blocks of 32; a sweep is the nb - 1 rounds of the round-robin
// pairing of the blocks, and a round diagonalises each of its nb / 2 pair
// subproblems (64 x 64, one CTA each, cyclic Jacobi in shared memory with the
// threshold rule) and applies the subproblems' rotations V to A (A <- P^T A P,
// P = the block-diagonal matrix of the V) and to the basis.
//
// Data movement: A is kept in the current round's layout, where pair q's two
// blocks sit at block positions 2q and 2q + 1, so a pair's rows form one
// contiguous panel.  A round is three launches:
//   solve   the pair subproblems (the diagonal 64 x 64 tiles) -> V, a flag;
//   rows T  X = V^T (A's pair panel), written transposed: A1 = (P^T A)^T =
//           A P (A is symmetric);
//   rows P  V^T (A1's pair panel) = P^T A P, written in the next round's
//           layout (rows and columns permuted), and the same product on the
//           basis panels Qt (rows = eigen-positions, columns = coordinates),
//           rows permuted.
// A pair whose subproblem needed no rotation copies its panel unchanged.
// Every sweep returns the blocks to round 0's layout; a sweep starts with the
// stopping rule (off-diagonal squared norm <= tol2 x the diagonal's), and a
// matrix that meets it is left alone from then on.  The last kernels read the
// eigenvalues off the diagonal, rank them, choose the signs against the
// previous basis and write the columns in rank order.
//
// Accuracy: the rotations are fp32 panel products with 64-deep sums; the
// threshold rule skips a pair whose off-diagonal entry is below tol2 / d of
// its diagonal product or below the level at which every entry together
// would meet the stopping rule (tol2 d2 / d^2, d2 the diagonal's squared
// norm), so entries at the rounding floor of a large row are not rotated
// again and again.
#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

namespace {

constexpr int kBjB = 32;            // block edge
constexpr int kBjP = 2 * kBjB;      // pair subproblem edge
constexpr int kBjPitch = kBjP + 1;  // odd pitch of the subproblem in shared memory
constexpr int kBjTile = 128;        // columns per CTA in the panel products
constexpr int kBjThreads = 256;
constexpr int kBjInner = 10;        // Jacobi sweeps per subproblem at most
constexpr int kBjParts = 32;        // fixed-slot partial sums of the stopping rule

__host__ __device__ inline int64_t r4(int64_t x) { return (x + 3) & ~int64_t(3); }

// per-matrix scratch, in floats
struct BjLayout {
  int64_t kk, v, a0, a1, q0, q1, vv, flags, lam, inv, orig, sign, parts, misc, total;
};

__host__ __device__ inline BjLayout bj_layout(int kp) {
  BjLayout L;
  const int64_t np = kp / kBjP;
  L.kk = static_cast<int64_t>(kp) * kp;
  L.a0 = 0;
  L.a1 = L.a0 + L.kk;
  L.q0 = L.a1 + L.kk;
  L.q1 = L.q0 + L.kk;
  L.vv = L.q1 + L.kk;
  L.flags = L.vv + np * kBjP * kBjP;
  L.lam = L.flags + r4(np);
  L.inv = L.lam + r4(kp);
  L.orig = L.inv + r4(kp);
  L.sign = L.orig + r4(kp);
  L.parts = L.sign + r4(kp);
  L.misc = L.parts + 4 * kBjParts;  // doubles: off, diag per part
  L.total = L.misc + 4;             // [0] done, [1] sweeps (ints), [2] d2 (float)
  L.v = 0;
  return L;
}

inline int bj_padded(int d) { return (d + kBjP - 1) / kBjP * kBjP; }

struct BjArgs {
  const float* A;      // count x d x d
  const float* Qh;     // count x d x d
  const float* Qprev;  // count x d x d
  float* Qout;         // count x d x d (may be Qprev)
  float* scratch;      // count x bj_layout(kp).total
  int d, kp, nb, count;
  float tol2;
  const uint32_t* status;
  uint32_t* status_w;
};

struct BjMat {
  float *a0, *a1, *q0, *q1, *vv, *lam, *sign;
  int *flags, *inv, *orig;
  double* parts;
  int* misc;
  float* d2;
};

__device__ __forceinline__ BjMat bj_mat(const BjArgs& P, int b) {
  const BjLayout L = bj_layout(P.kp);
  float* s = P.scratch + static_cast<int64_t>(b) * L.total;
  BjMat M;
  M.a0 = s + L.a0;
  M.a1 = s + L.a1;
  M.q0 = s + L.q0;
  M.q1 = s + L.q1;
  M.vv = s + L.vv;
  M.flags = reinterpret_cast<int*>(s + L.flags);
  M.lam = s + L.lam;
  M.inv = reinterpret_cast<int*>(s + L.inv);
  M.orig = reinterpret_cast<int*>(s + L.orig);
  M.sign = s + L.sign;
  M.parts = reinterpret_cast<double*>(s + L.parts);
  M.misc = reinterpret_cast<int*>(s + L.misc);
  M.d2 = s + L.misc + 2;
  return M;
}

// Round-robin pairing of nb blocks: in round rd the s-th slot holds block
// slot_block(s); pair q is (slot q, slot nb - 1 - q), stored at block
// positions 2q and 2q + 1.
__device__ __forceinline__ int slot_block(int s, int rd, int nb) { return s == 0 ? 0 : 1 + (s - 1 + rd) % (nb - 1); }

__device__ __forceinline__ int pos_block(int p, int rd, int nb) {
  const int q = p >> 1;
  return slot_block((p & 1) ? nb - 1 - q : q, rd, nb);
}

__device__ __forceinline__ int block_pos(int j, int rd, int nb) {
  const int s = j == 0 ? 0 : 1 + ((j - 1 - rd) % (nb - 1) + (nb - 1)) % (nb - 1);
  return s < nb / 2 ? 2 * s : 2 * (nb - 1 - s) + 1;
}

// the block position in round rd + 1's layout of the block at position p in
// round rd's
__device__ __forceinline__ int next_pos(int p, int rd, int nb) {
  return block_pos(pos_block(p, rd, nb), (rd + 1) % (nb - 1), nb);
}

__device__ __forceinline__ bool bj_skip(const BjArgs& P, const BjMat& M) {
  return __syncthreads_or(threadIdx.x == 0 &&
                          (*reinterpret_cast<const volatile uint32_t*>(P.status) != 0u ||
                           *reinterpret_cast<volatile int*>(M.misc) != 0));
}

__device__ __forceinline__ bool bj_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

// ------------------------------------------------------------------ setup
// A0 = round 0's layout of the symmetric part of A (zero padding); Qt0 = the
// rows of Q^^T in round 0's order (zero padding).  One 32 x 32 tile per CTA:
// blockIdx.z = 2 b + (0: A, 1: Qt).
__global__ void __launch_bounds__(kBjThreads) k_bj_init(BjArgs P) {
  __shared__ float t0[kBjB][kBjB + 1], t1[kBjB][kBjB + 1];
  const int b = blockIdx.z >> 1, what = blockIdx.z & 1;
  if (bj_flagged(P.status)) return;
  const BjMat M = bj_mat(P, b);
  const int d = P.d, kp = P.kp, nb = P.nb;
  const int pr = blockIdx.y, pc = blockIdx.x;  // destination block positions (what = 1: pc = coordinate block)
  const int br = pos_block(pr, 0, nb);
  const int64_t dd = static_cast<int64_t>(d) * d;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  if (what == 0) {
    const int bc = pos_block(pc, 0, nb);
    const float* Ab = P.A + b * dd;
    for (int r = ty; r < kBjB; r += 8) {
      const int i = br * kBjB + r, j = bc * kBjB + tx;
      t0[r][tx] = (i < d && j < d) ? Ab[static_cast<int64_t>(i) * d + j] : 0.0f;
      const int i2 = bc * kBjB + r, j2 = br * kBjB + tx;
      t1[r][tx] = (i2 < d && j2 < d) ? Ab[static_cast<int64_t>(i2) * d + j2] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < kBjB; r += 8)
      M.a0[static_cast<int64_t>(pr * kBjB + r) * kp + pc * kBjB + tx] = 0.5f * (t0[r][tx] + t1[tx][r]);
  } else {
    // Qt0[pr * 32 + r][c] = Q^[c][br * 32 + r], c in coordinate block pc
    const float* Qb = P.Qh + b * dd;
    for (int r = ty; r < kBjB; r += 8) {
      const int c = pc * kBjB + r, j = br * kBjB + tx;
      t0[r][tx] = (c < d && j < d) ? Qb[static_cast<int64_t>(c) * d + j] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < kBjB; r += 8)
      M.q0[static_cast<int64_t>(pr * kBjB + r) * kp + pc * kBjB + tx] = t0[tx][r];
  }
}

// --------------------------------------------------------- stopping rule
__global__ void __launch_bounds__(kBjThreads) k_bj_norms(BjArgs P) {
  __shared__ double red[2][kBjThreads / 32];
  const int b = blockIdx.y, part = blockIdx.x;
  const BjMat M = bj_mat(P, b);
  if (bj_skip(P, M)) return;
  const int kp = P.kp;
  const int rows = (kp + kBjParts - 1) / kBjParts;
  const int r0 = part * rows, r1 = min(kp, r0 + rows);
  double off = 0.0, dg = 0.0;
  for (int r = r0; r < r1; ++r) {
    const float* row = M.a0 + static_cast<int64_t>(r) * kp;
    for (int c = threadIdx.x; c < kp; c += blockDim.x) {
      const double v = row[c];
      if (c == r)
        dg += v * v;
      else
        off += v * v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    off += __shfl_xor_sync(0xffffffffu, off, o);
    dg += __shfl_xor_sync(0xffffffffu, dg, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = off;
    red[1][threadIdx.x >> 5] = dg;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double so = 0.0, sd = 0.0;
    for (int w = 0; w < kBjThreads / 32; ++w) {
      so += red[0][w];
      sd += red[1][w];
    }
    M.parts[2 * part] = so;
    M.parts[2 * part + 1] = sd;
  }
}

// one thread per matrix: the parts in order; done once the rule holds
__global__ void k_bj_decide(BjArgs P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.count) return;
  if (*reinterpret_cast<const volatile uint32_t*>(P.status) != 0u) return;
  const BjMat M = bj_mat(P, b);
  if (M.misc[0] != 0) return;
  double off = 0.0, dg = 0.0;
  for (int p = 0; p < kBjParts; ++p) {
    off += M.parts[2 * p];
    dg += M.parts[2 * p + 1];
  }
  if (!isfinite(off) || !isfinite(dg)) {
    atomicOr(P.status_w, kStNonfiniteIter);
    M.misc[0] = 1;
    return;
  }
  *M.d2 = static_cast<float>(dg);
  if (off <= static_cast<double>(P.tol2) * dg) {
    M.misc[0] = 1;
  } else {
    M.misc[1] += 1;  // sweeps run: the basis panels end in buffer (sweeps & 1)
  }
}

// ------------------------------------------------------------------ solve
// Pair q of round rd: the 64 x 64 diagonal tile of A0, diagonalised by cyclic
// Jacobi (threshold rule); V (row-major, columns = the rotated unit vectors)
// and a flag (any rotation) per pair.
__global__ void __launch_bounds__(kBjThreads) k_bj_solve(BjArgs P) {
  __shared__ float As[kBjP * kBjPitch];
  __shared__ float Vs[kBjP * kBjPitch];
  __shared__ float cs[kBjP];
  __shared__ int pr[kBjP];
  const int b = blockIdx.y, q = blockIdx.x;
  const BjMat M = bj_mat(P, b);
  if (bj_skip(P, M)) return;
  const int kp = P.kp;
  const float* T = M.a0 + static_cast<int64_t>(q) * kBjP * kp + q * kBjP;
  for (int e = threadIdx.x; e < kBjP * kBjP; e += blockDim.x) {
    const int i = e / kBjP, j = e % kBjP;
    As[i * kBjPitch + j] = 0.5f * (T[static_cast<int64_t>(i) * kp + j] + T[static_cast<int64_t>(j) * kp + i]);
    Vs[i * kBjPitch + j] = i == j ? 1.0f : 0.0f;
  }
  __syncthreads();
  const float t_rel = P.tol2 / static_cast<float>(P.d);
  const float t_abs = P.tol2 * (*M.d2) / (static_cast<float>(P.d) * static_cast<float>(P.d));
  bool any = false;
  for (int sweep = 0; sweep < kBjInner; ++sweep) {
    bool rot = false;
    for (int rd = 0; rd < kBjP - 1; ++rd) {
      if (threadIdx.x < kBjP / 2) {
        const int s = threadIdx.x;
        int pp = s == 0 ? 0 : 1 + (s - 1 + rd) % (kBjP - 1);
        const int s2 = kBjP - 1 - s;
        int qq = 1 + (s2 - 1 + rd) % (kBjP - 1);
        if (pp > qq) {
          const int x = pp;
          pp = qq;
          qq = x;
        }
        const float apq = As[pp * kBjPitch + qq];
        const float app = As[pp * kBjPitch + pp], aqq = As[qq * kBjPitch + qq];
        float c = 1.0f, sn = 0.0f;
        const float a2 = apq * apq;
        if (a2 > t_rel * fabsf(app * aqq) && a2 > t_abs) {
          const float th = (aqq - app) / (2.0f * apq);
          const float t = copysignf(1.0f, th) / (fabsf(th) + sqrtf(fmaf(th, th, 1.0f)));
          c = rsqrtf(fmaf(t, t, 1.0f));
          sn = t * c;
          rot = true;
        }
        cs[2 * s] = c;
        cs[2 * s + 1] = sn;
        pr[2 * s] = pp;
        pr[2 * s + 1] = qq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < (kBjP / 2) * kBjP; e += blockDim.x) {
        const int s = e / kBjP, j = e % kBjP;
        const float c = cs[2 * s], sn = cs[2 * s + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * s], qq = pr[2 * s + 1];
        const float ap = As[pp * kBjPitch + j], aq = As[qq * kBjPitch + j];
        As[pp * kBjPitch + j] = c * ap - sn * aq;
        As[qq * kBjPitch + j] = sn * ap + c * aq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < (kBjP / 2) * kBjP; e += blockDim.x) {
        const int s = e / kBjP, i = e % kBjP;
        const float c = cs[2 * s], sn = cs[2 * s + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * s], qq = pr[2 * s + 1];
        const float ap = As[i * kBjPitch + pp], aq = As[i * kBjPitch + qq];
        As[i * kBjPitch + pp] = c * ap - sn * aq;
        As[i * kBjPitch + qq] = sn * ap + c * aq;
        const float vp = Vs[i * kBjPitch + pp], vq = Vs[i * kBjPitch + qq];
        Vs[i * kBjPitch + pp] = c * vp - sn * vq;
        Vs[i * kBjPitch + qq] = sn * vp + c * vq;
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rot)) break;
    any = true;
  }
  if (threadIdx.x == 0) M.flags[q] = any ? 1 : 0;
  if (any) {
    // one polar step V (3 I - V^T V) / 2 takes the fp32 rounding of the
    // accumulated rotations off V's orthogonality (which the basis would
    // otherwise gather round after round); X = V^T V in the place of A
    float* Xs = As;
    for (int e = threadIdx.x; e < kBjP * kBjP; e += blockDim.x) {
      const int a = e / kBjP, c = e % kBjP;
      float x = 0.0f;
      for (int i = 0; i < kBjP; ++i) x = fmaf(Vs[i * kBjPitch + a], Vs[i * kBjPitch + c], x);
      Xs[a * kBjPitch + c] = (a == c ? 1.5f : 0.0f) - 0.5f * x;
    }
    __syncthreads();
    float* V = M.vv + static_cast<int64_t>(q) * kBjP * kBjP;
    for (int e = threadIdx.x; e < kBjP * kBjP; e += blockDim.x) {
      const int i = e / kBjP, c = e % kBjP;
      float v = 0.0f;
      for (int l = 0; l < kBjP; ++l) v = fmaf(Vs[i * kBjPitch + l], Xs[l * kBjPitch + c], v);
      V[e] = v;
    }
  }
}

// ------------------------------------------------------- panel products
// out (64 x 128) = V_q^T (src rows 64q.., columns c0..), or the panel itself
// when pair q was not rotated; written to dst as
//   mode 0: transposed, dst[c][64q + i]
//   mode 1: rows and columns moved to round rd + 1's block positions
//   mode 2: rows moved to round rd + 1's block positions
struct BjPanel {
  int src_buf, dst_buf, mode;  // buffers: 0 a0, 1 a1, 2 q0, 3 q1
};

__device__ __forceinline__ float* bj_buf(const BjMat& M, int i) {
  return i == 0 ? M.a0 : i == 1 ? M.a1 : i == 2 ? M.q0 : M.q1;
}

__global__ void __launch_bounds__(kBjThreads) k_bj_rows(BjArgs P, int rd, BjPanel t0, BjPanel t1, int ntarget) {
  __shared__ __align__(16) float sm[kBjP * kBjP + kBjP * kBjTile];  // V^T source, then the panel; reused for out
  const int b = blockIdx.z / ntarget, which = blockIdx.z % ntarget;
  const BjPanel T = which == 0 ? t0 : t1;
  const int q = blockIdx.y, c0 = blockIdx.x * kBjTile;
  const BjMat M = bj_mat(P, b);
  if (bj_skip(P, M)) return;
  const int kp = P.kp, nb = P.nb;
  const int ncol = min(kBjTile, kp - c0);  // a multiple of 64
  const float* src = bj_buf(M, T.src_buf);
  float* dst = bj_buf(M, T.dst_buf);
  const bool rotate = M.flags[q] != 0;
  float* Vs = sm;                    // [l][i], 64 x 64
  float* Is = sm + kBjP * kBjP;      // [l][c], 64 x 128
  const int tid = threadIdx.x;
  // the panel: 64 rows x ncol columns, float4 loads (zero past ncol)
  for (int f = tid; f < kBjP * kBjTile / 4; f += kBjThreads) {
    const int l = f / (kBjTile / 4), c4 = (f % (kBjTile / 4)) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < ncol)
      v = *reinterpret_cast<const float4*>(src + static_cast<int64_t>(q * kBjP + l) * kp + c0 + c4);
    *reinterpret_cast<float4*>(Is + l * kBjTile + c4) = v;
  }
  if (rotate) {
    const float* V = M.vv + static_cast<int64_t>(q) * kBjP * kBjP;
    for (int f = tid; f < kBjP * kBjP / 4; f += kBjThreads)
      *reinterpret_cast<float4*>(Vs + 4 * f) = *reinterpret_cast<const float4*>(V + 4 * f);
  }
  __syncthreads();
  // thread: rows 4 ti.., columns 8 tc..
  const int ti = tid >> 4, tc = tid & 15;
  float acc[4][8];
  if (rotate) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[u][v] = 0.0f;
#pragma unroll 4
    for (int l = 0; l < kBjP; ++l) {
      const float4 vv = *reinterpret_cast<const float4*>(Vs + l * kBjP + 4 * ti);
      const float4 x0 = *reinterpret_cast<const float4*>(Is + l * kBjTile + 8 * tc);
      const float4 x1 = *reinterpret_cast<const float4*>(Is + l * kBjTile + 8 * tc + 4);
      const float a[4] = {vv.x, vv.y, vv.z, vv.w};
      const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(a[u], x[v], acc[u][v]);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[u][v] = Is[(4 * ti + u) * kBjTile + 8 * tc + v];
  }
  __syncthreads();
  // stage out as [i][c] with an odd pitch, then write
  constexpr int kOp = kBjTile + 1;
  float* Os = sm;
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) Os[(4 * ti + u) * kOp + 8 * tc + v] = acc[u][v];
  __syncthreads();
  if (T.mode == 0) {
    // dst[c0 + c][64q + i]: 64 contiguous floats per column c
    for (int e = tid; e < ncol * kBjP; e += kBjThreads) {
      const int c = e / kBjP, i = e % kBjP;
      dst[static_cast<int64_t>(c0 + c) * kp + q * kBjP + i] = Os[i * kOp + c];
    }
  } else {
    // destination block positions: the pair's two row blocks, the tile's
    // column blocks (mode 1) or the columns as they are (mode 2)
    int* rmap = reinterpret_cast<int*>(sm + kBjP * kOp);  // past the staged output
    int* cmap = rmap + 2;
    if (tid < 2) rmap[tid] = next_pos(2 * q + tid, rd, nb);
    if (tid >= 32 && tid < 32 + kBjTile / kBjB) {
      const int cb = c0 / kBjB + (tid - 32);
      cmap[tid - 32] = T.mode == 1 && cb < nb ? next_pos(cb, rd, nb) : cb;
    }
    __syncthreads();
    for (int e = tid; e < kBjP * ncol; e += kBjThreads) {
      const int i = e / ncol, c = e % ncol;
      const int row = rmap[i / kBjB] * kBjB + (i & (kBjB - 1));
      const int col = cmap[c / kBjB] * kBjB + (c & (kBjB - 1));
      dst[static_cast<int64_t>(row) * kp + col] = Os[i * kOp + c];
    }
  }
}

// ----------------------------------------------------------------- finish
// ranks by decreasing eigenvalue (ties by original index) over the real
// positions of round 0's layout; inv[rank] = position
__global__ void __launch_bounds__(1024) k_bj_rank(BjArgs P) {
  const int b = blockIdx.x;
  if (bj_flagged(P.status)) return;
  const BjMat M = bj_mat(P, b);
  const int kp = P.kp, nb = P.nb, d = P.d;
  for (int p = threadIdx.x; p < kp; p += blockDim.x) {
    const int orig = pos_block(p / kBjB, 0, nb) * kBjB + (p & (kBjB - 1));
    M.orig[p] = orig;
    M.lam[p] = orig < d ? M.a0[static_cast<int64_t>(p) * kp + p] : 0.0f;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < kp; p += blockDim.x) {
    const int orig = M.orig[p];
    if (orig >= d) continue;
    const float lp = M.lam[p];
    int rank = 0;
    for (int p2 = 0; p2 < kp; ++p2) {
      const int o2 = M.orig[p2];
      const float l2 = M.lam[p2];
      rank += o2 < d && ((l2 > lp) || (l2 == lp && o2 < orig));
    }
    M.inv[rank] = p;
  }
}

// sign of column c: the product of the new column (row inv[c] of the basis
// panels) with column c of the previous basis; 32 columns per CTA
__global__ void __launch_bounds__(kBjThreads) k_bj_sign(BjArgs P) {
  __shared__ float tn[kBjB][kBjB + 1], tp[kBjB][kBjB + 1];
  __shared__ int rows[kBjB];
  const int b = blockIdx.y, c0 = blockIdx.x * kBjB;
  if (bj_flagged(P.status)) return;
  const BjMat M = bj_mat(P, b);
  const int d = P.d, kp = P.kp;
  const float* Qt = (M.misc[1] & 1) ? M.q1 : M.q0;
  const float* Qp = P.Qprev + static_cast<int64_t>(b) * d * d;
  if (threadIdx.x < kBjB) rows[threadIdx.x] = c0 + threadIdx.x < d ? M.inv[c0 + threadIdx.x] : -1;
  __syncthreads();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int cc = threadIdx.x >> 3, sub = threadIdx.x & 7;
  float dot = 0.0f;
  for (int i0 = 0; i0 < d; i0 += kBjB) {
    for (int r = ty; r < kBjB; r += 8) {
      const int row = rows[r], i = i0 + tx;
      tn[r][tx] = (row >= 0 && i < d) ? Qt[static_cast<int64_t>(row) * kp + i] : 0.0f;
      const int ii = i0 + r, c = c0 + tx;
      tp[r][tx] = (ii < d && c < d) ? Qp[static_cast<int64_t>(ii) * d + c] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = sub + 8 * u;
      dot = fmaf(tn[cc][i], tp[i][cc], dot);
    }
    __syncthreads();
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (sub == 0 && c0 + cc < d) M.sign[c0 + cc] = dot < 0.0f ? -1.0f : 1.0f;
}

// Qout[i][c] = sign[c] Qt[inv[c]][i]; 32 x 32 tiles
__global__ void __launch_bounds__(kBjThreads) k_bj_scatter(BjArgs P) {
  __shared__ float t[kBjB][kBjB + 1];
  const int b = blockIdx.z, c0 = blockIdx.x * kBjB, i0 = blockIdx.y * kBjB;
  if (bj_flagged(P.status)) return;
  const BjMat M = bj_mat(P, b);
  const int d = P.d, kp = P.kp;
  const float* Qt = (M.misc[1] & 1) ? M.q1 : M.q0;
  float* Qo = P.Qout + static_cast<int64_t>(b) * d * d;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < kBjB; r += 8) {
    const int c = c0 + r, i = i0 + tx;
    t[r][tx] = (c < d && i < d) ? M.sign[c] * Qt[static_cast<int64_t>(M.inv[c]) * kp + i] : 0.0f;
  }
  __syncthreads();
  for (int r = ty; r < kBjB; r += 8) {
    const int i = i0 + r, c = c0 + tx;
    if (i < d && c < d) Qo[static_cast<int64_t>(i) * d + c] = t[tx][r];
  }
}

__global__ void k_bj_reset(BjArgs P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.count) return;
  const BjMat M = bj_mat(P, b);
  M.misc[0] = 0;
  M.misc[1] = 0;
  *M.d2 = 0.0f;
}

}  // namespace

size_t bj_scratch_floats(int d) { return static_cast<size_t>(bj_layout(bj_padded(d)).total); }

cudaError_t launch_bjacobi(const BjSide& S, int max_sweeps, float tol2, uint32_t* status, cudaStream_t st,
                           int* launches) {
  if (S.count <= 0) return cudaSuccess;
  if (S.d <= kBjP || max_sweeps < 1 || !S.A || !S.Qh || !S.Qprev || !S.Qout || !S.scratch)
    return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(S.scratch) % 16 != 0) return cudaErrorInvalidValue;
  BjArgs P{};
  P.A = S.A;
  P.Qh = S.Qh;
  P.Qprev = S.Qprev;
  P.Qout = S.Qout;
  P.scratch = S.scratch;
  P.d = S.d;
  P.kp = bj_padded(S.d);
  P.nb = P.kp / kBjB;
  P.count = S.count;
  P.tol2 = tol2;
  P.status = status;
  P.status_w = status;
  const int nb = P.nb, np = nb / 2, count = S.count;
  const unsigned cnt = static_cast<unsigned>(count);
  int n = 0;
  k_bj_reset<<<(count + 127) / 128, 128, 0, st>>>(P);
  k_bj_init<<<dim3(nb, nb, 2 * cnt), kBjThreads, 0, st>>>(P);
  n += 2;
  const unsigned tiles = static_cast<unsigned>((P.kp + kBjTile - 1) / kBjTile);
  for (int s = 0; s < max_sweeps; ++s) {
    k_bj_norms<<<dim3(kBjParts, cnt), kBjThreads, 0, st>>>(P);
    k_bj_decide<<<(count + 127) / 128, 128, 0, st>>>(P);
    n += 2;
    for (int rd = 0; rd < nb - 1; ++rd) {
      // the basis panels alternate between q0 and q1 round by round
      const int g = s * (nb - 1) + rd;
      const BjPanel at{0, 1, 0};
      const BjPanel ap{1, 0, 1};
      const BjPanel qp{(g & 1) ? 3 : 2, (g & 1) ? 2 : 3, 2};
      k_bj_solve<<<dim3(np, cnt), kBjThreads, 0, st>>>(P);
      k_bj_rows<<<dim3(tiles, np, cnt), kBjThreads, 0, st>>>(P, rd, at, at, 1);
      k_bj_rows<<<dim3(tiles, np, 2 * cnt), kBjThreads, 0, st>>>(P, rd, ap, qp, 2);
      n += 3;
    }
  }
  const unsigned cb = static_cast<unsigned>((S.d + kBjB - 1) / kBjB);
  k_bj_rank<<<cnt, 1024, 0, st>>>(P);
  k_bj_sign<<<dim3(cb, cnt), kBjThreads, 0, st>>>(P);
  k_bj_scatter<<<dim3(cb, cb, cnt), kBjThreads, 0, st>>>(P);
  n += 3;
  if (launches) *launches += n;
  return cudaGetLastError();
}

}  // namespace okls

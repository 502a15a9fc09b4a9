// Blocked Jacobi eigensolver for the SOAP refresh past kClMaxK (sm_103a).
//
// Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
// Sketching", Appendix C, Algorithm 4 (SOAP): Eigenvectors(L, Q_L) -- the
// eigenvectors of the factor, ordered by decreasing eigenvalue, each column's
// sign matched to the previous basis.  The caller forms A = Q^^T F Q^ in the
// polar-corrected previous basis Q^; this file diagonalises A and writes
// Q^ W, reordered and sign-aligned, over the previous basis.
//
// The method: two-sided block Jacobi.  A (padded to kp, a multiple of 128,
// by zero rows and columns that no rotation ever touches) is split into
// nb = kp / 64 blocks of 64; a sweep is the nb - 1
// rounds of the round-robin pairing of the blocks, and a round diagonalises
// each of its nb / 2 pair subproblems (128 x 128, one CTA each, cyclic Jacobi
// in shared memory with the threshold rule, then one polar step on V) and
// applies the subproblems' rotations V to A (A <- P^T A P, P = the
// block-diagonal matrix of the V) and to the basis.
//
// Data movement: A is kept in the current round's layout, where pair q's two
// blocks sit at block positions 2q and 2q + 1, so a pair's rows form one
// contiguous panel.  A round is three launches:
//   solve   the pair subproblems (the diagonal 128 x 128 tiles) -> V, a flag;
//   rows T  X = V^T (A's pair panel), written transposed: A1 = (P^T A)^T =
//           A P (A is symmetric);
//   rows P  V^T (A1's pair panel) = P^T A P, written in the next round's
//           layout (rows and columns permuted), and the same product on the
//           basis panels Qt (rows = eigen-positions, columns = coordinates),
//           rows permuted.
// The panel products run on the tensor cores (okls_tc3.cu: three-term bf16
// split, fp32 accumulation; an identity V reproduces the panel exactly), or
// with OKLS_TC3=0 on the CUDA cores.  A pair whose subproblem needed no
// rotation copies its panel unchanged.
// Every sweep returns the blocks to round 0's layout; a sweep starts with the
// stopping rule (off-diagonal squared norm <= tol2 x the diagonal's), and a
// matrix that meets it is left alone from then on.  The last kernels read the
// eigenvalues off the diagonal, rank them, choose the signs against the
// previous basis and write the columns in rank order.
//
// Accuracy: the rotations are fp32-accurate panel products with 128-deep
// sums; the threshold rule skips a pair whose off-diagonal entry is below
// tol2 / d of its diagonal product or below the level at which every entry
// together would meet the stopping rule (tol2 d2 / d^2, d2 the diagonal's
// squared norm), so entries at the rounding floor of a large row are not
// rotated again and again.  After the sweeps the caller forms Q^T F Q anew
// from the basis found and runs up to two more sweeps on it (the tracked
// matrix gathers the rounding of hundreds of rounds).
#include <cuda_bf16.h>

#include <cstdlib>

#include "okls_bj.cuh"
#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

using namespace bj;

namespace {

constexpr int kT = 32;              // tile edge of the transposing copies
constexpr int kPitch = kP + 1;      // odd pitch of the subproblem in shared memory
constexpr int kSolveThreads = 512;
constexpr int kSolveSmem = 2 * kP * kPitch * 4 + kP * kP * 4;  // A, V, and the polar-corrected V
constexpr int kInner = 2;           // Jacobi sweeps per subproblem at most (more do not cut the outer sweeps; one is faster on small batches, slower on the 1.2B layer set)
constexpr int kThreads = 256;
constexpr int kRowCols = 64;        // columns per CTA of the CUDA-core panel product
constexpr int kRowSmem = (kP * kP + kP * kRowCols) * 4;

__device__ __forceinline__ bool flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

// ------------------------------------------------------------------ setup
// A0 = round 0's layout of the symmetric part of A (zero padding); Qt0 = the
// rows of Q^^T in round 0's order (zero padding).  One 32 x 32 tile per CTA:
// blockIdx.z = 2 b + (0: A, 1: Qt).
__global__ void __launch_bounds__(kThreads) k_bj_init(Args P) {
  __shared__ float t0[kT][kT + 1], t1[kT][kT + 1];
  const int b = blockIdx.z >> 1, what = blockIdx.z & 1;
  if (flagged(P.status)) return;
  const Mat M = mat(P, b);
  const int d = P.d, kp = P.kp, nb = P.nb;
  const int tr = blockIdx.y, tc = blockIdx.x;  // destination tile (what = 1: tc = coordinate tile)
  // the source rows of destination tile row tr: block pos_block(tr / 2), half tr % 2
  const int sr = pos_block(tr / 2, 0, nb) * kB + (tr & 1) * kT;
  const int64_t dd = static_cast<int64_t>(d) * d;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  if (what == 0) {
    const int sc = pos_block(tc / 2, 0, nb) * kB + (tc & 1) * kT;
    const float* Ab = P.A + b * dd;
    for (int r = ty; r < kT; r += 8) {
      const int i = sr + r, j = sc + tx;
      t0[r][tx] = (i < d && j < d) ? Ab[static_cast<int64_t>(i) * d + j] : 0.0f;
      const int i2 = sc + r, j2 = sr + tx;
      t1[r][tx] = (i2 < d && j2 < d) ? Ab[static_cast<int64_t>(i2) * d + j2] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < kT; r += 8)
      M.a0[static_cast<int64_t>(tr * kT + r) * kp + tc * kT + tx] = 0.5f * (t0[r][tx] + t1[tx][r]);
  } else {
    // Qt0[tr * 32 + r][c] = Q^[c][sr + r], c in coordinate tile tc
    const float* Qb = P.Qh + b * dd;
    for (int r = ty; r < kT; r += 8) {
      const int c = tc * kT + r, j = sr + tx;
      t0[r][tx] = (c < d && j < d) ? Qb[static_cast<int64_t>(c) * d + j] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < kT; r += 8)
      M.q0[static_cast<int64_t>(tr * kT + r) * kp + tc * kT + tx] = t0[tx][r];
  }
}

// --------------------------------------------------------- stopping rule
__global__ void __launch_bounds__(kThreads) k_bj_norms(Args P) {
  __shared__ double red[2][kThreads / 32];
  const int b = blockIdx.y, part = blockIdx.x;
  const Mat M = mat(P, b);
  if (skip(P, M)) return;
  const int kp = P.kp;
  const int rows = (kp + kParts - 1) / kParts;
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
    for (int w = 0; w < kThreads / 32; ++w) {
      so += red[0][w];
      sd += red[1][w];
    }
    M.parts[2 * part] = so;
    M.parts[2 * part + 1] = sd;
  }
}

// one thread per matrix: the parts in order; done once the rule holds
__global__ void k_bj_decide(Args P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.count) return;
  if (*reinterpret_cast<const volatile uint32_t*>(P.status) != 0u) return;
  const Mat M = mat(P, b);
  if (M.misc[0] != 0) return;
  double off = 0.0, dg = 0.0;
  for (int p = 0; p < kParts; ++p) {
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
// Pair q of the round: the 128 x 128 diagonal tile of A0, diagonalised by
// cyclic Jacobi (threshold rule), then one polar step on the accumulated
// rotations; V (row-major, columns = the rotated unit vectors) and a flag
// (any rotation) per pair.
__global__ void __launch_bounds__(kSolveThreads) k_bj_solve(Args P) {
  extern __shared__ float sm[];
  __shared__ float cs[kP];
  __shared__ int pr[kP];
  float* As = sm;
  float* Vs = sm + kP * kPitch;
  const int b = blockIdx.y, q = blockIdx.x;
  const Mat M = mat(P, b);
  if (skip(P, M)) return;
  const int kp = P.kp;
  const float* T = M.a0 + static_cast<int64_t>(q) * kP * kp + q * kP;
  for (int e = threadIdx.x; e < kP * kP; e += blockDim.x) {
    const int i = e / kP, j = e % kP;
    As[i * kPitch + j] = 0.5f * (T[static_cast<int64_t>(i) * kp + j] + T[static_cast<int64_t>(j) * kp + i]);
    Vs[i * kPitch + j] = i == j ? 1.0f : 0.0f;
  }
  __syncthreads();
  const float t_rel = P.tol2 / static_cast<float>(P.d);
  const float t_abs = P.tol2 * (*M.d2) / (static_cast<float>(P.d) * static_cast<float>(P.d));
  bool any = false;
  for (int sweep = 0; sweep < kInner; ++sweep) {
    bool rot = false;
    for (int rd = 0; rd < kP - 1; ++rd) {
      if (threadIdx.x < kP / 2) {
        const int s = threadIdx.x;
        int pp = s == 0 ? 0 : 1 + (s - 1 + rd) % (kP - 1);
        int qq = 1 + (kP - 2 - s + rd) % (kP - 1);  // slot kP - 1 - s (never 0)
        if (pp > qq) {
          const int x = pp;
          pp = qq;
          qq = x;
        }
        const float apq = As[pp * kPitch + qq];
        const float app = As[pp * kPitch + pp], aqq = As[qq * kPitch + qq];
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
      for (int e = threadIdx.x; e < (kP / 2) * kP; e += blockDim.x) {
        const int s = e / kP, j = e % kP;
        const float c = cs[2 * s], sn = cs[2 * s + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * s], qq = pr[2 * s + 1];
        const float ap = As[pp * kPitch + j], aq = As[qq * kPitch + j];
        As[pp * kPitch + j] = c * ap - sn * aq;
        As[qq * kPitch + j] = sn * ap + c * aq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < (kP / 2) * kP; e += blockDim.x) {
        const int s = e / kP, i = e % kP;
        const float c = cs[2 * s], sn = cs[2 * s + 1];
        if (sn == 0.0f) continue;
        const int pp = pr[2 * s], qq = pr[2 * s + 1];
        const float ap = As[i * kPitch + pp], aq = As[i * kPitch + qq];
        As[i * kPitch + pp] = c * ap - sn * aq;
        As[i * kPitch + qq] = sn * ap + c * aq;
        const float vp = Vs[i * kPitch + pp], vq = Vs[i * kPitch + qq];
        Vs[i * kPitch + pp] = c * vp - sn * vq;
        Vs[i * kPitch + qq] = sn * vp + c * vq;
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
    for (int e = threadIdx.x; e < kP * kP; e += blockDim.x) {
      const int a = e / kP, c = e % kP;
      float x = 0.0f;
      for (int i = 0; i < kP; ++i) x = fmaf(Vs[i * kPitch + a], Vs[i * kPitch + c], x);
      Xs[a * kPitch + c] = (a == c ? 1.5f : 0.0f) - 0.5f * x;
    }
    __syncthreads();
    float* Vc = sm + 2 * kP * kPitch;  // the corrected V, row-major
    float* V = M.vv + static_cast<int64_t>(q) * kP * kP;
    for (int e = threadIdx.x; e < kP * kP; e += blockDim.x) {
      const int i = e / kP, c = e % kP;
      float v = 0.0f;
      for (int l = 0; l < kP; ++l) v = fmaf(Vs[i * kPitch + l], Xs[l * kPitch + c], v);
      V[e] = v;
      Vc[e] = v;
    }
    __syncthreads();
    // V^T as the panel product's A operand (row r = i, k = l: V[l][i]), split
    // into three bf16 terms and laid out as the tensor core reads it: K-block
    // kb, term j, row r, 16-byte chunk kc at (kc ^ (r % 8)) * 16
    uint8_t* img = reinterpret_cast<uint8_t*>(M.vimg + static_cast<int64_t>(q) * kVimgFloats);
    constexpr int kPart = kP * 128;  // bytes of one term's image
    for (int e = threadIdx.x; e < kP * 2 * 8; e += blockDim.x) {
      const int r = e & (kP - 1), kc = (e >> 7) & 7, kb = e >> 10;
      uint32_t w[3][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int l = 64 * kb + 8 * kc + 2 * u;
        const float x0 = Vc[l * kP + r], x1 = Vc[(l + 1) * kP + r];
        const __nv_bfloat162 a = __floats2bfloat162_rn(x0, x1);
        const float r0 = x0 - __low2float(a), r1 = x1 - __high2float(a);
        const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
        const __nv_bfloat162 c = __floats2bfloat162_rn(r0 - __low2float(b), r1 - __high2float(b));
        w[0][u] = *reinterpret_cast<const uint32_t*>(&a);
        w[1][u] = *reinterpret_cast<const uint32_t*>(&b);
        w[2][u] = *reinterpret_cast<const uint32_t*>(&c);
      }
      const uint32_t off = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(kc) ^ (r & 7u)) << 4);
#pragma unroll
      for (int j = 0; j < 3; ++j)
        *reinterpret_cast<uint4*>(img + (kb * 3 + j) * kPart + off) = make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]);
    }
  }
}

// ------------------------------------------- panel products on the CUDA cores
// out (128 x 64) = V_q^T (src rows 128q.., columns c0..c0+63), or the panel
// itself when pair q was not rotated; written to dst by the panel's mode.
__global__ void __launch_bounds__(kThreads) k_bj_rows(Args P, int rd, Panel t0, Panel t1, int ntarget) {
  extern __shared__ __align__(16) float rs[];  // V (128 x 128), then the panel (128 x 64); reused for out
  const int b = blockIdx.z / ntarget, which = blockIdx.z % ntarget;
  const Panel T = which == 0 ? t0 : t1;
  const int q = blockIdx.y, c0 = blockIdx.x * kRowCols;
  const Mat M = mat(P, b);
  if (skip(P, M)) return;
  const int kp = P.kp, nb = P.nb;
  const float* src = buf(M, T.src_buf);
  float* dst = buf(M, T.dst_buf);
  const bool rotate = M.flags[q] != 0;
  float* Vs = rs;               // [l][i]
  float* Is = rs + kP * kP;     // [l][c]
  const int tid = threadIdx.x;
  for (int f = tid; f < kP * kRowCols / 4; f += kThreads) {
    const int l = f / (kRowCols / 4), c4 = (f % (kRowCols / 4)) * 4;
    *reinterpret_cast<float4*>(Is + l * kRowCols + c4) =
        *reinterpret_cast<const float4*>(src + static_cast<int64_t>(q * kP + l) * kp + c0 + c4);
  }
  if (rotate) {
    const float* V = M.vv + static_cast<int64_t>(q) * kP * kP;
    for (int f = tid; f < kP * kP / 4; f += kThreads)
      *reinterpret_cast<float4*>(Vs + 4 * f) = *reinterpret_cast<const float4*>(V + 4 * f);
  }
  __syncthreads();
  // thread: rows 8 ti.., columns 4 tc..
  const int ti = tid >> 4, tc = tid & 15;
  float acc[8][4];
  if (rotate) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
#pragma unroll 4
    for (int l = 0; l < kP; ++l) {
      const float4 a0 = *reinterpret_cast<const float4*>(Vs + l * kP + 8 * ti);
      const float4 a1 = *reinterpret_cast<const float4*>(Vs + l * kP + 8 * ti + 4);
      const float4 x = *reinterpret_cast<const float4*>(Is + l * kRowCols + 4 * tc);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], xv[v], acc[u][v]);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = Is[(8 * ti + u) * kRowCols + 4 * tc + v];
  }
  __syncthreads();
  // stage out as [i][c] with an odd pitch, then write
  constexpr int kOp = kRowCols + 1;
  float* Os = rs;
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) Os[(8 * ti + u) * kOp + 4 * tc + v] = acc[u][v];
  __syncthreads();
  if (T.mode == 0) {
    // dst[c0 + c][128q + i]: 128 contiguous floats per column c
    for (int e = tid; e < kRowCols * kP; e += kThreads) {
      const int c = e / kP, i = e % kP;
      dst[panel_dst(0, q, i, c0 + c, rd, nb, kp)] = Os[i * kOp + c];
    }
  } else {
    for (int e = tid; e < kP * kRowCols; e += kThreads) {
      const int i = e / kRowCols, c = e % kRowCols;
      dst[panel_dst(T.mode, q, i, c0 + c, rd, nb, kp)] = Os[i * kOp + c];
    }
  }
}

// ----------------------------------------------------------------- finish
// ranks by decreasing eigenvalue (ties by original index) over the real
// positions of round 0's layout; inv[rank] = position
__global__ void __launch_bounds__(1024) k_bj_rank(Args P) {
  const int b = blockIdx.x;
  if (flagged(P.status)) return;
  const Mat M = mat(P, b);
  const int kp = P.kp, nb = P.nb, d = P.d;
  for (int p = threadIdx.x; p < kp; p += blockDim.x) {
    const int orig = pos_block(p / kB, 0, nb) * kB + (p & (kB - 1));
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
__global__ void __launch_bounds__(kThreads) k_bj_sign(Args P) {
  __shared__ float tn[kT][kT + 1], tp[kT][kT + 1];
  __shared__ int rows[kT];
  const int b = blockIdx.y, c0 = blockIdx.x * kT;
  if (flagged(P.status)) return;
  const Mat M = mat(P, b);
  const int d = P.d, kp = P.kp;
  const float* Qt = (M.misc[1] & 1) ? M.q1 : M.q0;
  const float* Qp = P.Qprev + static_cast<int64_t>(b) * d * d;
  if (threadIdx.x < kT) rows[threadIdx.x] = c0 + threadIdx.x < d ? M.inv[c0 + threadIdx.x] : -1;
  __syncthreads();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int cc = threadIdx.x >> 3, sub = threadIdx.x & 7;
  float dot = 0.0f;
  for (int i0 = 0; i0 < d; i0 += kT) {
    for (int r = ty; r < kT; r += 8) {
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
__global__ void __launch_bounds__(kThreads) k_bj_scatter(Args P) {
  __shared__ float t[kT][kT + 1];
  const int b = blockIdx.z, c0 = blockIdx.x * kT, i0 = blockIdx.y * kT;
  if (flagged(P.status)) return;
  const Mat M = mat(P, b);
  const int d = P.d, kp = P.kp;
  const float* Qt = (M.misc[1] & 1) ? M.q1 : M.q0;
  float* Qo = P.Qout + static_cast<int64_t>(b) * d * d;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < kT; r += 8) {
    const int c = c0 + r, i = i0 + tx;
    t[r][tx] = (c < d && i < d) ? M.sign[c] * Qt[static_cast<int64_t>(M.inv[c]) * kp + i] : 0.0f;
  }
  __syncthreads();
  for (int r = ty; r < kT; r += 8) {
    const int i = i0 + r, c = c0 + tx;
    if (i < d && c < d) Qo[static_cast<int64_t>(i) * d + c] = t[tx][r];
  }
}

__global__ void k_bj_reset(Args P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.count) return;
  const Mat M = mat(P, b);
  M.misc[0] = 0;
  M.misc[1] = 0;
  *M.d2 = 0.0f;
}

bool tc_panels() {
  static const int on = [] {
    const char* e = getenv("OKLS_TC3");
    return (e && e[0] == '0') ? 0 : 1;
  }();
  return on != 0;
}

}  // namespace

size_t bj_scratch_floats(int d) { return static_cast<size_t>(layout(padded(d)).total); }

cudaError_t launch_bjacobi(const BjSide& S, int max_sweeps, float tol2, uint32_t* status, cudaStream_t st,
                           int* launches) {
  if (S.count <= 0) return cudaSuccess;
  if (S.d <= kB || max_sweeps < 1 || !S.A || !S.Qh || !S.Qprev || !S.Qout || !S.scratch)
    return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(S.scratch) % 16 != 0) return cudaErrorInvalidValue;
  static PerDevice pd;
  cudaError_t e = once_per_device(pd, [](int) {
    cudaError_t r = cudaFuncSetAttribute(k_bj_solve, cudaFuncAttributeMaxDynamicSharedMemorySize, kSolveSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(k_bj_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowSmem);
    return r;
  });
  if (e != cudaSuccess) return e;
  Args P{};
  P.A = S.A;
  P.Qh = S.Qh;
  P.Qprev = S.Qprev;
  P.Qout = S.Qout;
  P.scratch = S.scratch;
  P.d = S.d;
  P.kp = padded(S.d);
  P.nb = P.kp / kB;
  P.count = S.count;
  P.tol2 = tol2;
  P.status = status;
  P.status_w = status;
  const int nb = P.nb, np = nb / 2, count = S.count;
  const unsigned cnt = static_cast<unsigned>(count);
  const bool tc = tc_panels();
  int n = 0;
  k_bj_reset<<<(count + 127) / 128, 128, 0, st>>>(P);
  const unsigned tiles32 = static_cast<unsigned>(P.kp / kT);
  k_bj_init<<<dim3(tiles32, tiles32, 2 * cnt), kThreads, 0, st>>>(P);
  n += 2;
  const unsigned row_tiles = static_cast<unsigned>(P.kp / kRowCols);
  for (int s = 0; s < max_sweeps; ++s) {
    k_bj_norms<<<dim3(kParts, cnt), kThreads, 0, st>>>(P);
    k_bj_decide<<<(count + 127) / 128, 128, 0, st>>>(P);
    n += 2;
    for (int rd = 0; rd < nb - 1; ++rd) {
      // the basis panels alternate between q0 and q1 round by round
      const int g = s * (nb - 1) + rd;
      const Panel at{0, 1, 0};
      const Panel ap{1, 0, 1};
      const Panel qp{(g & 1) ? 3 : 2, (g & 1) ? 2 : 3, 2};
      k_bj_solve<<<dim3(np, cnt), kSolveThreads, kSolveSmem, st>>>(P);
      if (tc) {
        e = launch_t3_panels(P, rd, at, at, 1, st);
        if (e == cudaSuccess) e = launch_t3_panels(P, rd, ap, qp, 2, st);
        if (e != cudaSuccess) return e;
      } else {
        k_bj_rows<<<dim3(row_tiles, np, cnt), kThreads, kRowSmem, st>>>(P, rd, at, at, 1);
        k_bj_rows<<<dim3(row_tiles, np, 2 * cnt), kThreads, kRowSmem, st>>>(P, rd, ap, qp, 2);
      }
      n += 3;
    }
  }
  const unsigned cb = static_cast<unsigned>((S.d + kT - 1) / kT);
  k_bj_rank<<<cnt, 1024, 0, st>>>(P);
  k_bj_sign<<<dim3(cb, cnt), kThreads, 0, st>>>(P);
  k_bj_scatter<<<dim3(cb, cb, cnt), kThreads, 0, st>>>(P);
  n += 3;
  if (launches) *launches += n;
  return cudaGetLastError();
}

}  // namespace okls

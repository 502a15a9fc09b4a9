// Batched symmetric eigensolver for k x k matrices, 128 < k <= kClMaxK
// (sm_103a): cyclic Jacobi with the rotations of each sweep logged and
// applied to the eigenvector matrix by a separate, wide kernel.
//
// Used by the SOAP refresh (Clean page, Appendix C, Algorithm 4:
// Eigenvectors(L, Q_L)) and by Clean's thin SVD of the sketch (Clean page,
// Appendix A, Algorithm 3: the eigen-decomposition of Z^T Z).
//
// Per sweep, two launches:
//   sweep        the sweep's stopping rule, then the dp - 1 rounds of the
//                round-robin ordering: each computes its dp / 2 disjoint
//                rotations (threshold Jacobi: a pair whose off-diagonal entry
//                is already below tol2 / k of its diagonal is left alone),
//                writes them to the sweep's log and applies J^T A J as one
//                pass over the 2 x 2 blocks of every two pairs.  Two kernels:
//                k_eig_sweep_l2 keeps A as a full symmetric dp x dp matrix in
//                an L2-resident workspace slice and runs each matrix on a
//                thread-block cluster of 1, 2, 4 or 8 CTAs (every access of a
//                round is a contiguous run of a row); k_eig_sweep_packed keeps
//                A as a packed triangle in one CTA's shared memory (k <= 330).
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
#include <cstdlib>

#include "okls_internal.h"
#include "okls_kernels.h"

namespace okls {

namespace {

constexpr int kEigPackMaxK = 330;  // packed triangle in shared memory up to here
constexpr int kEigThreads = 1024;
constexpr int kApplyRows = 32;
constexpr int kApplyPitch = kApplyRows + 4;  // floats per column of a band (16-byte rows, banks staggered)
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

// One sweep on one matrix per CTA with A as a packed triangle in shared
// memory (k <= kEigPackMaxK), loaded from / stored to the slice around the
// sweep.
__device__ void sweep_packed(const EigPlan& P, const EigSide& S, int b, int sweep, float* sm) {
  __shared__ float red[kEigThreads / 32];
  const int k = S.k;
  const int dp = k + (k & 1), np = dp / 2;
  const EigSlice sl = eig_slice(S.scratch, k, b);
  // a converged matrix stays converged: later sweeps do nothing
  if (sweep > 0 && sl.flags[0] == 0) {
    if (threadIdx.x == 0) sl.flags[1] = 0;
    return;
  }
  float* cs = sm;                                      // 2 per pair
  int* pr = reinterpret_cast<int*>(sm + 2 * kClMaxK);  // 2 per pair
  float* A = sm + kEigHead;
  const int tid = threadIdx.x, nth = blockDim.x;
  const int npk = dp * (dp + 1) / 2;
  if (sweep == 0) {
    // the symmetric part of the input, padded by a zero row and column when k is odd
    const float* G = S.A + static_cast<int64_t>(b) * k * k;
    for (int j = tid; j < dp; j += nth)
      for (int i = 0; i <= j; ++i) A[pk(i, j, dp)] = (i < k && j < k) ? 0.5f * (G[i * k + j] + G[j * k + i]) : 0.0f;
  } else {
    for (int e = tid; e < npk; e += nth) A[e] = sl.A[e];
  }
  __syncthreads();
  float off = 0.0f, dg = 0.0f;
  for (int j = tid; j < dp; j += nth)
    for (int i = 0; i <= j; ++i) {
      const float v = A[pk(i, j, dp)];
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
        const float2 r = jacobi_cs(A[pk(pp, pp, dp)], A[pk(qq, qq, dp)], A[pk(pp, qq, dp)], skip2);
        cs[2 * q] = r.x;
        cs[2 * q + 1] = r.y;
        pr[2 * q] = pp;
        pr[2 * q + 1] = qq;
        sl.log[static_cast<int64_t>(rd) * np + q] = r;
      }
      __syncthreads();
      // the upper blocks (u <= v)
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
      __syncthreads();
    }
  }
  // back to the slice for the next sweep and the finishing kernel (at sweep
  // 0 also when nothing rotated: it was built here)
  if (more || sweep == 0)
    for (int e = tid; e < npk; e += nth) sl.A[e] = A[e];
}

__global__ void __launch_bounds__(kEigThreads) k_eig_sweep_packed(const __grid_constant__ EigPlan P, int sweep) {
  extern __shared__ float sm[];
  if (eig_flagged(P.status)) return;
  const Where w = locate(P, 1, 1);
  sweep_packed(P, *w.side, w.b, sweep, sm);
}

__device__ __forceinline__ unsigned cl_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cl_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; global writes before it are
// visible to the cluster's reads after it
__device__ __forceinline__ void cl_barrier(unsigned nc) {
  if (nc > 1)
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  else
    __syncthreads();
}

// The L2 pass's block item (x, y): load its four entries (false when the
// item is out of range or both its rotations are the identity) ...
__device__ __forceinline__ bool l2_load(const float* A, int dp, const float2* cs, const int2* pr, int x, int y, int np,
                                        Blk& c) {
  if (y >= np) return false;
  if (cs[x].y == 0.0f && cs[y].y == 0.0f) return false;
  const int2 px = pr[x], py = pr[y];
  const float* r1 = A + px.x * dp;
  const float* r2 = A + px.y * dp;
  c = Blk{__ldcg(r1 + py.x), __ldcg(r1 + py.y), __ldcg(r2 + py.x), __ldcg(r2 + py.y)};
  return true;
}

// ... and store its rotated entries.  The block of the unordered pair is
// formed from the lower index's rows: for x > y that is C^T, and the result
// is written transposed.
__device__ __forceinline__ void l2_store(float* A, int dp, const float2* cs, const int2* pr, int x, int y,
                                         const Blk c) {
  const float2 cx = cs[x], cy = cs[y];
  const int2 px = pr[x], py = pr[y];
  float* r1 = A + px.x * dp;
  float* r2 = A + px.y * dp;
  if (x == y) {
    const Blk n = rot2(c, cx.x, cx.y, cx.x, cx.y);
    __stcg(r1 + px.x, n.a11);
    __stcg(r1 + px.y, n.a12);
    __stcg(r2 + px.x, n.a12);
    __stcg(r2 + px.y, n.a22);
  } else {
    const bool tr = x > y;
    const Blk in = tr ? Blk{c.a11, c.a21, c.a12, c.a22} : c;
    const float2 lo = tr ? cy : cx, hi = tr ? cx : cy;
    const Blk n = rot2(in, lo.x, lo.y, hi.x, hi.y);
    __stcg(r1 + py.x, n.a11);
    __stcg(r1 + py.y, tr ? n.a21 : n.a12);
    __stcg(r2 + py.x, tr ? n.a12 : n.a21);
    __stcg(r2 + py.y, n.a22);
  }
}

__device__ __forceinline__ void next_task(int& xg, int& yg, int dxg, int dyg, int ng) {
  xg += dxg;
  yg += dyg;
  if (yg >= ng) {
    yg -= ng;
    ++xg;
  }
}

// One sweep with A as a full symmetric dp x dp matrix in the L2-resident
// slice, on a cluster of nc CTAs per matrix (nc = 1: a plain launch).  CTA c
// of the cluster applies the blocks of the row pairs x in its share of
// [0, dp / 2); every CTA forms all of a round's rotations itself (the same
// numbers in each), and two cluster barriers per round separate the reads of
// the rotation inputs from the pass's writes and the pass from the next
// round.  A is read through L2 (ld.global.cg): other SMs write it.
__global__ void __launch_bounds__(kEigThreads) k_eig_sweep_l2(const __grid_constant__ EigPlan P, int sweep) {
  extern __shared__ float sm[];
  __shared__ float red[kEigThreads / 32];
  const unsigned nc = cl_size(), rank = cl_rank();
  if (eig_flagged(P.status)) return;
  const Where w = locate(P, static_cast<int>(nc), static_cast<int>(nc));
  const EigSide& S = *w.side;
  const int k = S.k, b = w.b;
  const int dp = k + (k & 1), np = dp / 2;
  const EigSlice sl = eig_slice(S.scratch, k, b);
  if (sweep > 0 && __ldcg(sl.flags) == 0) {
    if (rank == 0 && threadIdx.x == 0) sl.flags[1] = 0;
    return;
  }
  float2* cs = reinterpret_cast<float2*>(sm);               // per pair
  int2* pr = reinterpret_cast<int2*>(sm + 2 * kClMaxK);     // per pair
  float* A = sl.A;
  const int tid = threadIdx.x, nth = blockDim.x;
  if (sweep == 0) {
    const float* G = S.A + static_cast<int64_t>(b) * k * k;
    for (int j = static_cast<int>(rank) * nth + tid; j < dp; j += static_cast<int>(nc) * nth)
      for (int i = 0; i <= j; ++i) {
        const float v = (i < k && j < k) ? 0.5f * (G[i * k + j] + G[j * k + i]) : 0.0f;
        __stcg(A + i * dp + j, v);
        __stcg(A + j * dp + i, v);
      }
    cl_barrier(nc);
  }
  float off = 0.0f, dg = 0.0f;
  for (int j = tid; j < dp; j += nth)
#pragma unroll 4
    for (int i = 0; i <= j; ++i) {
      const float v = __ldcg(A + i * dp + j);
      if (i == j)
        dg = fmaf(v, v, dg);
      else
        off = fmaf(2.0f * v, v, off);
    }
  const float offs = eig_block_sum(off, red);
  const float dgs = eig_block_sum(dg, red);
  // every CTA of the cluster reached the same decision from the same sums;
  // the flags change only after all of them have read them
  const bool more = offs > P.tol2 * dgs;
  cl_barrier(nc);
  if (rank == 0 && tid == 0) {
    sl.flags[0] = more ? 1 : 0;
    sl.flags[1] = more ? 1 : 0;
  }
  if (!more) return;
  const float skip2 = P.tol2 / static_cast<float>(k);
  const int x0 = static_cast<int>(rank) * np / static_cast<int>(nc);
  const int x1 = (static_cast<int>(rank) + 1) * np / static_cast<int>(nc);
  const int ng = (np + 31) >> 5;   // groups of 32 column pairs
  const int nx = x1 - x0;
  const int warp = tid >> 5, lane = tid & 31, nwarp = nth >> 5;
  // task counters (row pair, column group), advanced by nwarp tasks at a time
  const int xg0 = warp / ng, yg0 = warp - (warp / ng) * ng;
  const int dxg = nwarp / ng, dyg = nwarp - (nwarp / ng) * ng;
  for (int rd = 0; rd < dp - 1; ++rd) {
    for (int q = tid; q < np; q += nth) {
      int pp, qq;
      round_pair(q, rd, dp, pp, qq);
      const float2 r = jacobi_cs(__ldcg(A + pp * dp + pp), __ldcg(A + qq * dp + qq), __ldcg(A + pp * dp + qq), skip2);
      cs[q] = r;
      pr[q] = make_int2(pp, qq);
      if (rank == 0) sl.log[static_cast<int64_t>(rd) * np + q] = r;
    }
    __syncthreads();
    cl_barrier(nc);
    // task = (row pair x, 32 column pairs y); x is the same on every lane.
    // Two tasks per iteration: both tasks' loads are in flight together.
    int xg = xg0, yg = yg0;
    while (xg < nx) {
      int xg2 = xg, yg2 = yg;
      next_task(xg2, yg2, dxg, dyg, ng);
      const int xa = x0 + xg, ya = (yg << 5) + lane;
      const int xb = x0 + xg2, yb = (yg2 << 5) + lane;
      Blk ca, cb;
      const bool acta = l2_load(A, dp, cs, pr, xa, ya, np, ca);
      const bool actb = xg2 < nx && l2_load(A, dp, cs, pr, xb, yb, np, cb);
      if (acta) l2_store(A, dp, cs, pr, xa, ya, ca);
      if (actb) l2_store(A, dp, cs, pr, xb, yb, cb);
      next_task(xg2, yg2, dxg, dyg, ng);
      xg = xg2;
      yg = yg2;
    }
    cl_barrier(nc);
  }
}

// V <- V J for the rotations logged by sweep `sweep`, on a band of
// kApplyRows rows of V per CTA (V = I before sweep 0).  The band sits in
// shared memory column by column (pitch kApplyPitch), so that a rotation
// moves four rows per 16-byte access; rows past the band's end are zeros
// and are rotated along without being stored.
__global__ void __launch_bounds__(kApplyThreads) k_eig_apply(const __grid_constant__ EigPlan P, int sweep,
                                                            int bands0, int bands1) {
  extern __shared__ float4 vs4[];
  float* vs = reinterpret_cast<float*>(vs4);
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
    vs[j * kApplyPitch + r] = v;
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
          float4* cp = vs4 + pp * (kApplyPitch / 4);
          float4* cq = vs4 + qq * (kApplyPitch / 4);
#pragma unroll
          for (int r4 = 0; r4 < kApplyRows / 4; ++r4) {
            const float4 a = cp[r4], b = cq[r4];
            cp[r4] = make_float4(fmaf(c, a.x, -(sn * b.x)), fmaf(c, a.y, -(sn * b.y)), fmaf(c, a.z, -(sn * b.z)),
                                 fmaf(c, a.w, -(sn * b.w)));
            cq[r4] = make_float4(fmaf(sn, a.x, c * b.x), fmaf(sn, a.y, c * b.y), fmaf(sn, a.z, c * b.z),
                                 fmaf(sn, a.w, c * b.w));
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
    sl.V[static_cast<int64_t>(l0 + r) * k + j] = vs[j * kApplyPitch + r];
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
  const bool full = S.full != 0;
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
  static PerDevice pd;
  return once_per_device(pd, [](int) {
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(k_eig_sweep_packed, at, sweep_smem(kEigPackMaxK));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_eig_apply, at, kApplyPitch * kClMaxK * 4);
    return e;
  });
}

cudaLaunchConfig_t l2_config(int nb, int nc, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(nb * nc));
  cfg.blockDim = dim3(kEigThreads);
  cfg.dynamicSmemBytes = kEigHead * 4;
  cfg.stream = st;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = static_cast<unsigned>(nc);
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nc > 1 ? 1 : 0;
  return cfg;
}

// CTAs per matrix for the L2 sweep: 8, 4 or 2 where every matrix's cluster
// is resident at once (cluster sizes that leave part of the grid to a second
// wave measured slower than one CTA per matrix), else 1
int cluster_size(int nb) {
  static PerDevice pd;
  static int active[64][9];  // per device: co-resident clusters of each size
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 1;
  once_per_device(pd, [](int d) {
    for (int nc = 2; nc <= 8; nc *= 2) {
      cudaLaunchAttribute attr;
      cudaLaunchConfig_t cfg = l2_config(1, nc, nullptr, &attr);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(k_eig_sweep_l2), &cfg) != cudaSuccess)
        n = 0;
      active[d][nc] = n;
    }
    (void)cudaGetLastError();
    return cudaSuccess;
  });
  int cap = 8;
  // OKLS_EIG_CTAS=c caps the CTAs per matrix (tests run the one-CTA kernels
  // on small batches with c = 1)
  if (const char* env = getenv("OKLS_EIG_CTAS")) {
    const int c = atoi(env);
    if (c >= 1) cap = std::min(cap, c);
  }
  for (int nc = 8; nc >= 2; nc /= 2)
    if (nc <= cap && nb <= active[dev][nc]) return nc;
  return 1;
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
  const int nc = cluster_size(nb);
  int smem = 0, dpmax = 0, bands[2] = {1, 1}, napply = 0;
  bool any_large = false;
  for (int i = 0; i < 2; ++i) {
    const EigSide& S = P.side[i];
    if (S.count == 0) continue;
    any_large |= S.k > kEigPackMaxK;
    smem = std::max(smem, sweep_smem(S.k));
    dpmax = std::max(dpmax, S.k + (S.k & 1));
    bands[i] = (S.k + kApplyRows - 1) / kApplyRows;
    napply += S.count * bands[i];
  }
  // one CTA per matrix with A in shared memory where that fits, unless
  // clusters of 4 or more CTAs per matrix fit at once (measured: 1.4-1.6x
  // faster at k = 256-320 with 4); clusters over A in L2 past 330 (every
  // side alike, so that one launch covers both)
  const bool l2 = nc >= 4 || any_large;
  const int ncl = l2 ? nc : 1;
  EigPlan Q = P;
  Q.side[0].full = Q.side[1].full = l2 ? 1 : 0;
  const int apply_smem = kApplyPitch * dpmax * 4;
  for (int s = 0; s < Q.max_sweeps; ++s) {
    if (l2) {
      cudaLaunchAttribute attr;
      const cudaLaunchConfig_t cfg = l2_config(nb, ncl, st, &attr);
      e = cudaLaunchKernelEx(&cfg, k_eig_sweep_l2, Q, s);
      if (e != cudaSuccess) return e;
    } else {
      k_eig_sweep_packed<<<nb, kEigThreads, smem, st>>>(Q, s);
    }
    k_eig_apply<<<napply, kApplyThreads, apply_smem, st>>>(Q, s, bands[0], bands[1]);
  }
  k_eig_finish<<<nb, kFinishThreads, 0, st>>>(Q);
  if (launches) *launches += 2 * Q.max_sweeps + 1;
  return cudaGetLastError();
}

}  // namespace okls

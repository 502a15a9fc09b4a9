// Bandwidth-bound kernels of the OKLS step (sm_103a).
//
//   k_momentum_stats  M_t = b1 M + (1-b1) G and N_t = kappa (b1 M_t + (1-b1) G)
//                     evaluated on the fly to get sum G^2, sum N^2 per matrix
//                     (page "Online KL Shampoo": Nesterov momentum with
//                     variance correction); flags non-finite inputs.
//   k_coeffs_pre      per-matrix power-of-two scales of G and N and the EMA
//                     weights of both factors (the plain-sum weights of the
//                     classic Shampoo factors in that mode).
//   k_pack            writes M_t, Ghat, Nhat and Ghat^T (binary16, scaled);
//                     the transpose goes through 32x32 shared-memory tiles.
//   k_coeffs_post     normaliser c' of each factor and the chain's output
//                     scales; after the chain the root scales pi; the
//                     whitening coefficient.
//   k_normalise       Y_0 = (S + rho c I)/c', T_0 = a_0 I + b_0 Y_0, Z_1 = T_0
//                     (the first Newton-Schulz step needs no product).
//   k_sumsq, k_amax, k_requant, k_reset_state: inverse-root entry and state
//                     management.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "okls_internal.h"
#include "okls_kernels.h"
#include "okls_norm.cuh"

namespace okls {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.0f;
  if (w == 0) {
    s = (l < static_cast<int>(blockDim.x >> 5)) ? red[l] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  return s;  // valid in thread 0
}

// ------------------------------------------------------------ momentum stats
// 8 consecutive elements of G (bf16 or fp32) and of M as floats
template <typename GT>
__device__ __forceinline__ void load8(const GT* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

// Sums of G^2 and N^2 of one matrix per blockIdx.y, one fixed partial per
// block.  kVec: 8 elements per thread and step with 16-byte loads (mn a
// multiple of 8, so every matrix starts 16-byte aligned).
template <typename GT, bool kVec>
__global__ void k_momentum_stats(const GT* __restrict__ G, const float* __restrict__ M,
                                 int64_t mn, float b1, float kappa, float* part, int64_t part_ld,
                                 int batch, uint32_t* status) {
  __shared__ float red[32];
  const int b = blockIdx.y;
  const GT* g = G + static_cast<int64_t>(b) * mn;
  const float* mo = M ? M + static_cast<int64_t>(b) * mn : nullptr;  // null: no momentum
  float sg = 0.0f, sn = 0.0f;
  bool bad = false;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (kVec) {
    for (int64_t e8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e8 < mn / 8; e8 += stride) {
      float gv[8], mv[8];
      load8<GT>(g + e8 * 8, gv);
      if (mo) {
        load8<float>(mo + e8 * 8, mv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) mv[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float mn1 = fmaf(b1, mv[e], (1.0f - b1) * gv[e]);
        const float nv = kappa * fmaf(b1, mn1, (1.0f - b1) * gv[e]);
        bad |= !isfinite(gv[e]) || !isfinite(mv[e]);
        sg = fmaf(gv[e], gv[e], sg);
        sn = fmaf(nv, nv, sn);
      }
    }
  } else {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < mn; e += stride) {
      const float gv = to_f(g[e]);
      const float mv = mo ? mo[e] : 0.0f;
      const float mn1 = fmaf(b1, mv, (1.0f - b1) * gv);
      const float nv = kappa * fmaf(b1, mn1, (1.0f - b1) * gv);
      bad |= !isfinite(gv) || !isfinite(mv);
      sg = fmaf(gv, gv, sg);
      sn = fmaf(nv, nv, sn);
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kStNonfiniteInput);
  const float tg = block_sum(sg, red);
  const float tn = block_sum(sn, red);
  // per-block partials in fixed slots: [0: G, 1: N][batch][block]
  if (threadIdx.x == 0) {
    part[static_cast<int64_t>(b) * part_ld + blockIdx.x] = tg;
    part[(static_cast<int64_t>(batch) + b) * part_ld + blockIdx.x] = tn;
  }
}

// Double sum of n partials by one warp in a fixed order: lane l adds
// p[l], p[l+32], ... in turn, then the lanes' sums are combined by a fixed
// butterfly and lane 0's value is broadcast, so every run gives the same bits.
__device__ __forceinline__ double warp_sum_parts(const float* p, int64_t n) {
  const int lane = threadIdx.x & 31;
  double s = 0.0;
  for (int64_t i = lane; i < n; i += 32) s += static_cast<double>(p[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return __shfl_sync(0xffffffffu, s, 0);
}
constexpr int kCoeffWarps = 4;  // matrices per block of the coefficient kernels

// power of two 2^e with rms * 2^e in [1, 2); 1 for an all-zero matrix
__device__ __forceinline__ float pow2_rms_scale(float sumsq, double count) {
  const float r = static_cast<float>(sqrt(static_cast<double>(sumsq) / count));
  if (!(r > 0.0f) || !isfinite(r)) return 1.0f;
  int e = -ilogbf(r);
  e = max(-100, min(100, e));
  return ldexpf(1.0f, e);
}

// one warp per matrix
__global__ void k_coeffs_pre(int batch, int64_t m, int64_t n, float beta2, int shampoo, float* scal,
                             int scal_ld, const float* part, int64_t part_ld, int nparts) {
  const int b = blockIdx.x * kCoeffWarps + (threadIdx.x >> 5);
  if (b >= batch) return;
  const double sg = warp_sum_parts(part + static_cast<int64_t>(b) * part_ld, nparts);
  const double sn = warp_sum_parts(part + (static_cast<int64_t>(batch) + b) * part_ld, nparts);
  if ((threadIdx.x & 31) != 0) return;
  auto S = [&](int slot) -> float& { return scal[static_cast<int64_t>(slot) * scal_ld + b]; };
  S(SC_SUMSQ_G) = static_cast<float>(sg);
  S(SC_SUMSQ_N) = static_cast<float>(sn);
  const double cnt = static_cast<double>(m) * static_cast<double>(n);
  const float gs = pow2_rms_scale(S(SC_SUMSQ_G), cnt);
  const float ns = pow2_rms_scale(S(SC_SUMSQ_N), cnt);
  S(SC_GSCALE) = gs;
  S(SC_NSCALE) = ns;
  if (shampoo) {
    // L += G G^T = Ghat Ghat^T / gs^2 (and R likewise): weight 1, no roots
    const double w = 1.0 / (static_cast<double>(gs) * gs);
    S(SC_ALPHA_SA) = static_cast<float>(w);
    S(SC_ALPHA_SB) = static_cast<float>(w);
    return;
  }
  // X_b = G P_b = Xhat_b 2^h pi_b / gs  ->  S_a += (1-b2)/n (2^h pi_b / gs)^2 Xhat Xhat^T
  const double h = ldexp(1.0, kHeadroom);
  const double xa = h * S(SC_PI_B) / gs;
  const double xb = h * S(SC_PI_A) / gs;
  S(SC_ALPHA_SA) = static_cast<float>((1.0 - beta2) / static_cast<double>(n) * xa * xa);
  S(SC_ALPHA_SB) = static_cast<float>((1.0 - beta2) / static_cast<double>(m) * xb * xb);
}

// ------------------------------------------------------------------ pack
// One block per 64 x 64 tile of one matrix: 8 threads cover a 64-column row,
// 8 consecutive columns each (16-byte loads and stores when n is a multiple
// of 8); M_t, Ghat and Nhat go out row-major, and Ghat^T through the
// shared-memory tile, again 8 consecutive entries per thread.
constexpr int kPT = 64;

template <typename GT>
__global__ void __launch_bounds__(256) k_pack(const GT* __restrict__ G, float* __restrict__ M,
                                              __half* __restrict__ Gh, __half* __restrict__ GhT,
                                              __half* __restrict__ Nh, int m, int n, int64_t ldm, int64_t ldn,
                                              float b1, float kappa, const float* scal, int scal_ld,
                                              const uint32_t* status) {
  __shared__ float sg[kPT][kPT + 1];
  if (*reinterpret_cast<const volatile uint32_t*>(status) != 0u) return;
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * kPT, c0 = blockIdx.x * kPT;
  const float gs = scal[static_cast<int64_t>(SC_GSCALE) * scal_ld + b];
  const float ns = scal[static_cast<int64_t>(SC_NSCALE) * scal_ld + b];
  const int64_t mn = static_cast<int64_t>(m) * n;
  const GT* g = G + b * mn;
  float* mo = M ? M + b * mn : nullptr;  // null: no momentum (Shampoo)
  __half* gh = Gh + b * static_cast<int64_t>(m) * ldn;
  __half* nh = Nh ? Nh + b * static_cast<int64_t>(m) * ldn : nullptr;  // null: N = G
  const bool vec = (n & 7) == 0;
  // rows r0 + R: 8 threads cover 64 columns, 8 each (16-byte loads/stores)
#pragma unroll 1
  for (int p = 0; p < kPT / 32; ++p) {
    const int R = p * 32 + threadIdx.x / 8, C = (threadIdx.x % 8) * 8;
    const int i = r0 + R, j = c0 + C;
    float gv[8], mv[8], nv[8];
    const bool full = vec && i < m && j + 8 <= n;
    if (full) {
      load8<GT>(g + static_cast<int64_t>(i) * n + j, gv);
      if (mo) load8<float>(mo + static_cast<int64_t>(i) * n + j, mv);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool in = i < m && j + e < n;
        gv[e] = in ? to_f(g[static_cast<int64_t>(i) * n + j + e]) : 0.0f;
        mv[e] = (in && mo) ? mo[static_cast<int64_t>(i) * n + j + e] : 0.0f;
      }
    }
    if (!mo) {
#pragma unroll
      for (int e = 0; e < 8; ++e) mv[e] = 0.0f;
    }
    __align__(16) __half hg[8], hn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float m1 = fmaf(b1, mv[e], (1.0f - b1) * gv[e]);
      nv[e] = kappa * fmaf(b1, m1, (1.0f - b1) * gv[e]);
      mv[e] = m1;
      hg[e] = __float2half_rn(gv[e] * gs);
      hn[e] = __float2half_rn(nv[e] * ns);
      sg[R][C + e] = gv[e] * gs;
    }
    if (full) {
      if (mo) {
        float4* dm = reinterpret_cast<float4*>(mo + static_cast<int64_t>(i) * n + j);
        dm[0] = make_float4(mv[0], mv[1], mv[2], mv[3]);
        dm[1] = make_float4(mv[4], mv[5], mv[6], mv[7]);
      }
      *reinterpret_cast<uint4*>(gh + static_cast<int64_t>(i) * ldn + j) = *reinterpret_cast<const uint4*>(hg);
      if (nh) *reinterpret_cast<uint4*>(nh + static_cast<int64_t>(i) * ldn + j) = *reinterpret_cast<const uint4*>(hn);
    } else if (i < m) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (j + e < n) {
          if (mo) mo[static_cast<int64_t>(i) * n + j + e] = mv[e];
          gh[static_cast<int64_t>(i) * ldn + j + e] = hg[e];
          if (nh) nh[static_cast<int64_t>(i) * ldn + j + e] = hn[e];
        }
      }
    }
  }
  __syncthreads();
  // Ghat^T: row c0 + R holds column R of the tile; 8 threads per 64 entries
  __half* gt = GhT + b * static_cast<int64_t>(n) * ldm;
#pragma unroll 1
  for (int p = 0; p < kPT / 32; ++p) {
    const int R = p * 32 + threadIdx.x / 8, C = (threadIdx.x % 8) * 8;
    const int jt = c0 + R, i0 = r0 + C;
    if (jt >= n) continue;
    __align__(16) __half ht[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) ht[e] = __float2half_rn(sg[C + e][R]);
    if (i0 + 8 <= m) {
      *reinterpret_cast<uint4*>(gt + static_cast<int64_t>(jt) * ldm + i0) = *reinterpret_cast<const uint4*>(ht);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (i0 + e < m) gt[static_cast<int64_t>(jt) * ldm + i0 + e] = ht[e];
    }
  }
}

// -------------------------------------------------------------- post scalars
// mode bits: kPostRoots   c' and the chain's output scales from ||S||_F (before a chain)
//            kPostCommit  pi of the new roots (after the chain, so a chain that
//                         failed leaves P^ and pi of the previous roots together)
//            kPostUpdate  the whitening coefficient from pi_a, pi_b and N's scale
__global__ void k_coeffs_post(int batch, float ridge, int zK, int zK1, float* scal, int scal_ld, int mode,
                              const uint32_t* status, const float* part_a, int64_t part_a_ld, int64_t npart_a,
                              const float* part_b, int64_t part_b_ld, int64_t npart_b) {
  // one warp per matrix
  const int b = blockIdx.x * kCoeffWarps + (threadIdx.x >> 5);
  if (b >= batch) return;
  // a failed stage leaves the previous roots (and their scales) in force
  if (*reinterpret_cast<const volatile uint32_t*>(status) != 0u) return;
  // ||S||_F^2 of both factors from their fixed partial slots
  const double sa = part_a ? warp_sum_parts(part_a + b * part_a_ld, npart_a) : 0.0;
  const double sb = part_b ? warp_sum_parts(part_b + b * part_b_ld, npart_b) : 0.0;
  if ((threadIdx.x & 31) != 0) return;
  auto S = [&](int slot) -> float& { return scal[static_cast<int64_t>(slot) * scal_ld + b]; };
  if (part_a) S(SC_SUMSQ_SA) = static_cast<float>(sa);
  if (part_b) S(SC_SUMSQ_SB) = static_cast<float>(sb);
  const double margin = 1.0 + ldexp(1.0, -8);
  const int h = kHeadroom;
  for (int f = 0; f < 2 && (mode & kPostRoots); ++f) {
    const int s_sum = f == 0 ? SC_SUMSQ_SA : SC_SUMSQ_SB;
    double c = sqrt(static_cast<double>(S(s_sum)));
    double cp = c * (1.0 + ridge) * margin;
    if (!(cp > 1e-30)) cp = 1e-30;
    const double rc = 1.0 / sqrt(cp);
    S(f == 0 ? SC_CPRIME_A : SC_CPRIME_B) = static_cast<float>(cp);
    S(f == 0 ? SC_PSCALE_A : SC_PSCALE_B) = static_cast<float>(ldexp(rc, zK1 - 2 * h));
    S(f == 0 ? SC_RSCALE_A : SC_RSCALE_B) = static_cast<float>(ldexp(sqrt(cp), -2 * h));
  }
  for (int f = 0; f < 2 && (mode & kPostCommit); ++f) {
    const double cp = static_cast<double>(S(f == 0 ? SC_CPRIME_A : SC_CPRIME_B));
    S(f == 0 ? SC_PI_A : SC_PI_B) = static_cast<float>(ldexp(1.0 / sqrt(cp), zK - h));
  }
  if (mode & kPostUpdate) {
    const double pa = S(SC_PI_A), pb = S(SC_PI_B), ns = S(SC_NSCALE);
    S(SC_UCOEF) = static_cast<float>(ldexp(pa * pb / ns, h));
  }
}

// ---------------------------------------------------------------- normalise
// One block per pair of 64 x 64 tiles (tr, tc), tr <= tc, of one matrix: S is
// read once per pair (the upper tile, or both tiles when a full input is
// symmetrised), the outputs of the upper tile are written row by row and
// those of the mirrored tile (equal by symmetry, recomputed bit for bit from
// the same fp32 value) from the transposed shared-memory tile, and for
// upper-only input the lower tile of S is written back as the mirror.
constexpr int kNT = 64;         // normaliser tile edge
constexpr int kNTP = kNT + 1;   // padded shared-memory pitch

// the q-th (tr, tc) of the upper triangle of an nt x nt tile grid, row-major
__device__ __forceinline__ void upper_pair(int q, int nt, int& tr, int& tc) {
  // reversed index u counts from the last row, whose rows hold 1, 2, ... tiles
  const int u = nt * (nt + 1) / 2 - 1 - q;
  int k = static_cast<int>((sqrtf(8.0f * static_cast<float>(u) + 1.0f) - 1.0f) * 0.5f);
  while (k * (k + 1) / 2 > u) --k;
  while ((k + 1) * (k + 2) / 2 <= u) ++k;
  tr = nt - 1 - k;
  tc = nt - 1 - (u - k * (k + 1) / 2);
}

__device__ __forceinline__ NormOut norm_value(const NormaliseArgs& A, float s, bool diag, float inv, float rc,
                                             float a0h, float zsc) {
  return norm_value_core(s, diag, inv, rc, a0h, A.b0, zsc, A.split_y != 0, A.split_t != 0, A.split_z != 0);
}

// Write the outputs of 8 consecutive columns [j0, j0+8) of row i (binary16
// rows are 16-byte aligned; ragged ends fall back to single stores).
__device__ __forceinline__ void norm_store8(const NormaliseArgs& A, int64_t moff, int i, int j0, int d,
                                           const float* v, float inv, float rc, float a0h, float zsc, bool& bad) {
  __align__(16) __half hy[8], ht[8], hz[8], ly[8], lt[8], lz[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const NormOut o = norm_value(A, v[e], j0 + e == i, inv, rc, a0h, zsc);
    hy[e] = o.y;
    ht[e] = o.t;
    hz[e] = o.z;
    ly[e] = o.yl;
    lt[e] = o.tl;
    lz[e] = o.zl;
    bad |= o.bad && (j0 + e < d);
  }
  const int64_t e0 = moff + static_cast<int64_t>(i) * A.ld16 + j0;
  if (j0 + 8 <= d) {
    *reinterpret_cast<uint4*>(A.Y + e0) = *reinterpret_cast<const uint4*>(hy);
    *reinterpret_cast<uint4*>(A.T + e0) = *reinterpret_cast<const uint4*>(ht);
    *reinterpret_cast<uint4*>(A.Z + e0) = *reinterpret_cast<const uint4*>(hz);
    if (A.split_y) *reinterpret_cast<uint4*>(A.Ylo + e0) = *reinterpret_cast<const uint4*>(ly);
    if (A.split_t) *reinterpret_cast<uint4*>(A.Tlo + e0) = *reinterpret_cast<const uint4*>(lt);
    if (A.split_z) *reinterpret_cast<uint4*>(A.Zlo + e0) = *reinterpret_cast<const uint4*>(lz);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (j0 + e < d) {
        A.Y[e0 + e] = hy[e];
        A.T[e0 + e] = ht[e];
        A.Z[e0 + e] = hz[e];
        if (A.split_y) A.Ylo[e0 + e] = ly[e];
        if (A.split_t) A.Tlo[e0 + e] = lt[e];
        if (A.split_z) A.Zlo[e0 + e] = lz[e];
      }
    }
  }
}

__global__ void __launch_bounds__(256, 3) k_normalise(NormaliseArgs A) {
  __shared__ float sm[kNT][kNTP];
  // this grid raises the status word itself: one read per block keeps the
  // early exit uniform across the block's threads
  if (A.status && __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(A.status) != 0u))
    return;
  const int b = blockIdx.y;
  const int d = A.d;
  const int nt = (d + kNT - 1) / kNT;
  int tr, tc;
  upper_pair(static_cast<int>(blockIdx.x), nt, tr, tc);
  const int r0 = tr * kNT, c0 = tc * kNT;
  const bool diag_tile = tr == tc;
  float* S = A.S + static_cast<int64_t>(b) * d * d;
  const int tid = threadIdx.x;
  const bool vec = (d & 3) == 0;

  // 1. the upper tile (r0.., c0..) into shared memory; a full input is
  //    symmetrised with its transposed tile, (S + S^T) / 2
  for (int q = tid; q < kNT * (kNT / 4); q += 256) {
    const int r = q / (kNT / 4), c = (q % (kNT / 4)) * 4;
    const int i = r0 + r, j = c0 + c;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (i < d) {
      const float* src = S + static_cast<int64_t>(i) * d + j;
      if (vec && j + 3 < d) {
        v = *reinterpret_cast<const float4*>(src);
      } else {
        if (j < d) v.x = src[0];
        if (j + 1 < d) v.y = src[1];
        if (j + 2 < d) v.z = src[2];
        if (j + 3 < d) v.w = src[3];
      }
    }
    sm[r][c] = v.x;
    sm[r][c + 1] = v.y;
    sm[r][c + 2] = v.z;
    sm[r][c + 3] = v.w;
  }
  __syncthreads();
  if (!A.upper_only) {
    // add the tile (c0.., r0..) transposed; on the diagonal tile that is the
    // tile itself
    float part[16];
    const int r = tid / 4, cb = (tid % 4) * 16;  // this thread's 16 entries of row r of the tile
    if (diag_tile) {
#pragma unroll
      for (int e = 0; e < 16; ++e) part[e] = 0.5f * (sm[r][cb + e] + sm[cb + e][r]);
    } else {
      // S[c0 + cb + e][r0 + r]: a column of the lower tile, read once per entry
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int i2 = c0 + cb + e, j2 = r0 + r;
        const float w = (i2 < d && j2 < d) ? S[static_cast<int64_t>(i2) * d + j2] : 0.0f;
        part[e] = 0.5f * (sm[r][cb + e] + w);
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 16; ++e) sm[r][cb + e] = part[e];
    __syncthreads();
  } else if (diag_tile) {
    // upper-only diagonal tile: the entries below the diagonal are the mirror
    float part[16];
    const int r = tid / 4, cb = (tid % 4) * 16;
#pragma unroll
    for (int e = 0; e < 16; ++e) part[e] = (cb + e >= r) ? sm[r][cb + e] : sm[cb + e][r];
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 16; ++e) sm[r][cb + e] = part[e];
    __syncthreads();
  }

  // 2. the lower triangle of the state for upper-only input: rows c0 + R of
  //    the lower tile hold sm[.][R]; 16 threads write one 256-byte row
  if (A.upper_only) {
#pragma unroll 1
    for (int p = 0; p < kNT / 16; ++p) {
      const int R = p * 16 + tid / 16, C = (tid % 16) * 4;
      const int i = c0 + R, j = r0 + C;
      if (i >= d) continue;
      float* dst = S + static_cast<int64_t>(i) * d + j;
      const float v0 = sm[C][R], v1 = sm[C + 1][R], v2 = sm[C + 2][R], v3 = sm[C + 3][R];
      if (!diag_tile && vec && j + 3 < d) {
        *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
      } else {
        // the diagonal tile writes only below the diagonal
        if (j < d && (!diag_tile || j < i)) dst[0] = v0;
        if (j + 1 < d && (!diag_tile || j + 1 < i)) dst[1] = v1;
        if (j + 2 < d && (!diag_tile || j + 2 < i)) dst[2] = v2;
        if (j + 3 < d && (!diag_tile || j + 3 < i)) dst[3] = v3;
      }
    }
  }
  if (A.mirror_only) return;

  // 3. Y_0, T_0, Z_1 of the upper tile, then of the mirrored tile; 8 threads
  //    cover one 128-byte binary16 row of the tile
  const float cp = A.scal[static_cast<int64_t>(A.slot_cprime) * A.scal_ld + b];
  const float c = sqrtf(A.scal[static_cast<int64_t>(A.slot_sumsq) * A.scal_ld + b]);
  const float inv = ldexpf(1.0f, kHeadroom) / cp;
  const float rc = A.ridge * c;
  const float a0h = ldexpf(A.a0, kHeadroom);
  const float zsc = ldexpf(1.0f, -A.z1);
  const int64_t moff = static_cast<int64_t>(b) * A.mat16;
  bool bad = false;
#pragma unroll 1
  for (int p = 0; p < kNT / 32; ++p) {
    const int R = p * 32 + tid / 8, C = (tid % 8) * 8;
    {
      const int i = r0 + R;
      if (i < d && c0 + C < d) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = sm[R][C + e];
        norm_store8(A, moff, i, c0 + C, d, v, inv, rc, a0h, zsc, bad);
      }
    }
    if (!diag_tile) {
      const int i = c0 + R;
      if (i < d && r0 + C < d) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = sm[C + e][R];
        norm_store8(A, moff, i, r0 + C, d, v, inv, rc, a0h, zsc, bad);
      }
    }
  }
  if (bad && A.status) atomicOr(A.status, kStNonfiniteIter);
}

// ------------------------------------------------------------- small helpers
__global__ void k_sumsq(const float* __restrict__ S, int64_t dd, float* part, int64_t part_ld) {
  __shared__ float red[32];
  const int b = blockIdx.y;
  const float* s = S + static_cast<int64_t>(b) * dd;
  float acc = 0.0f;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < dd;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    acc = fmaf(s[e], s[e], acc);
  const float t = block_sum(acc, red);
  if (threadIdx.x == 0) part[static_cast<int64_t>(b) * part_ld + blockIdx.x] = t;
}

__global__ void k_amax(const float* __restrict__ P, int64_t dd, float* scal, int scal_ld, int slot) {
  __shared__ float red[32];
  const int b = blockIdx.y;
  const float* p = P + static_cast<int64_t>(b) * dd;
  float acc = 0.0f;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < dd;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    acc = fmaxf(acc, fabsf(p[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = fmaxf(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = 0.0f;
    for (int q = 0; q < static_cast<int>(blockDim.x >> 5); ++q) mx = fmaxf(mx, red[q]);
    // non-negative floats order like their bit patterns
    atomicMax(reinterpret_cast<unsigned int*>(scal + static_cast<int64_t>(slot) * scal_ld + b),
              __float_as_uint(mx));
  }
}

// pi = 2^(ceil(log2 amax) - h); the amax slot is overwritten by pi.
__global__ void k_requant_scale(int batch, float* scal, int scal_ld, int slot) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  float& s = scal[static_cast<int64_t>(slot) * scal_ld + b];
  const float amax = s;
  int e = 0;
  if (amax > 0.0f && isfinite(amax)) {
    e = ilogbf(amax);
    if (ldexpf(1.0f, e) < amax) ++e;
  }
  s = ldexpf(1.0f, e - kHeadroom);
}

// Phat = P / pi (row-major and transposed, 32x32 tiles); optional lo halves
__global__ void k_requant(const float* __restrict__ P, int d, __half* Ph, __half* PhT, __half* Pl,
                          __half* PlT, int64_t ld16, int64_t mat16, const float* scal, int scal_ld, int slot) {
  __shared__ float t[32][33];
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const float inv = 1.0f / scal[static_cast<int64_t>(slot) * scal_ld + b];
  const float* p = P + static_cast<int64_t>(b) * d * d;
  const int tx = threadIdx.x;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int i = r0 + r, j = c0 + tx;
    float v = 0.0f;
    if (i < d && j < d) {
      v = p[static_cast<int64_t>(i) * d + j] * inv;
      const __half hv = __float2half_rn(v);
      Ph[b * mat16 + static_cast<int64_t>(i) * ld16 + j] = hv;
      if (Pl) Pl[b * mat16 + static_cast<int64_t>(i) * ld16 + j] = __float2half_rn(v - __half2float(hv));
    }
    t[r][tx] = v;
  }
  __syncthreads();
  for (int c = threadIdx.y; c < 32; c += 8) {
    const int j = c0 + c, i = r0 + tx;
    if (i < d && j < d) {
      const float v = t[tx][c];
      const __half hv = __float2half_rn(v);
      if (PhT) PhT[b * mat16 + static_cast<int64_t>(j) * ld16 + i] = hv;
      if (PlT) PlT[b * mat16 + static_cast<int64_t>(j) * ld16 + i] = __float2half_rn(v - __half2float(hv));
    }
  }
}

// M = 0, S = eps I, P = I; Phat = 2^h I (pi = 2^-h), low halves 0
__global__ void k_reset_factor(float* S, float* P, __half* Ph, __half* PhT, __half* Pl, __half* PlT, int d,
                               int64_t ld16, int64_t mat16, int batch, float eps) {
  const int64_t dd = static_cast<int64_t>(d) * d;
  const int64_t tot = dd * batch;
  const __half one = __float2half_rn(ldexpf(1.0f, kHeadroom));
  const __half zero = __float2half_rn(0.0f);
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < tot;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = e / dd, r = e % dd;
    const int64_t i = r / d, j = r % d;
    const bool diag = i == j;
    S[e] = diag ? eps : 0.0f;
    P[e] = diag ? 1.0f : 0.0f;
    const int64_t o = b * mat16 + i * ld16 + j;
    Ph[o] = diag ? one : zero;
    if (PhT) PhT[o] = diag ? one : zero;
    if (Pl) Pl[o] = zero;
    if (PlT) PlT[o] = zero;
  }
}

__global__ void k_fill_scal(float* scal, int scal_ld, int slot, int batch, float v) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) scal[static_cast<int64_t>(slot) * scal_ld + b] = v;
}

// ---------------------------------------------------------------- launchers
static int grid_for(int64_t n, int per_block, int cap) {
  int64_t g = (n + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

int momentum_parts(int64_t mn) { return grid_for(mn, 256 * 8, kMaxStatParts); }

cudaError_t launch_momentum_stats(const void* G, int g_bf16, const float* M, int batch, int64_t mn,
                                  float b1, float kappa, float* part, int64_t part_ld, uint32_t* status,
                                  cudaStream_t st) {
  const int per_mat = momentum_parts(mn);
  if (per_mat > part_ld) return cudaErrorInvalidValue;
  dim3 grid(per_mat, batch);
  const bool vec = (mn % 8) == 0;
  if (g_bf16) {
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(G);
    if (vec)
      k_momentum_stats<__nv_bfloat16, true><<<grid, 256, 0, st>>>(g, M, mn, b1, kappa, part, part_ld, batch, status);
    else
      k_momentum_stats<__nv_bfloat16, false><<<grid, 256, 0, st>>>(g, M, mn, b1, kappa, part, part_ld, batch, status);
  } else {
    const float* g = static_cast<const float*>(G);
    if (vec)
      k_momentum_stats<float, true><<<grid, 256, 0, st>>>(g, M, mn, b1, kappa, part, part_ld, batch, status);
    else
      k_momentum_stats<float, false><<<grid, 256, 0, st>>>(g, M, mn, b1, kappa, part, part_ld, batch, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_coeffs_pre(int batch, int64_t m, int64_t n, float beta2, int shampoo, float* scal,
                              int scal_ld, const float* part, int64_t part_ld, cudaStream_t st) {
  k_coeffs_pre<<<(batch + kCoeffWarps - 1) / kCoeffWarps, 32 * kCoeffWarps, 0, st>>>(batch, m, n, beta2, shampoo,
                                                                                     scal, scal_ld, part, part_ld,
                                                    momentum_parts(m * n));
  return cudaGetLastError();
}

cudaError_t launch_pack(const void* G, int g_bf16, float* M, __half* Gh, __half* GhT, __half* Nh,
                        int batch, int m, int n, int64_t ldm, int64_t ldn, float b1, float kappa,
                        const float* scal, int scal_ld, const uint32_t* status, cudaStream_t st) {
  dim3 grid((n + kPT - 1) / kPT, (m + kPT - 1) / kPT, batch);
  if (g_bf16)
    k_pack<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(G), M, Gh, GhT, Nh, m, n, ldm,
                                                ldn, b1, kappa, scal, scal_ld, status);
  else
    k_pack<float><<<grid, 256, 0, st>>>(static_cast<const float*>(G), M, Gh, GhT, Nh, m, n, ldm, ldn, b1, kappa,
                                        scal, scal_ld, status);
  return cudaGetLastError();
}

cudaError_t launch_coeffs_post(int batch, float ridge, int zK, int zK1, float* scal, int scal_ld, int mode,
                               const uint32_t* status, const float* part_a, int64_t part_a_ld, int64_t npart_a,
                               const float* part_b, int64_t part_b_ld, int64_t npart_b, cudaStream_t st) {
  k_coeffs_post<<<(batch + kCoeffWarps - 1) / kCoeffWarps, 32 * kCoeffWarps, 0, st>>>(batch, ridge, zK, zK1, scal,
                                                                                      scal_ld, mode, status, part_a,
                                                     part_a_ld, npart_a, part_b, part_b_ld, npart_b);
  return cudaGetLastError();
}

cudaError_t launch_normalise(const NormaliseArgs& A, int batch, cudaStream_t st) {
  const int nt = (A.d + kNT - 1) / kNT;
  dim3 grid(nt * (nt + 1) / 2, batch);
  k_normalise<<<grid, 256, 0, st>>>(A);
  return cudaGetLastError();
}

int sumsq_parts(int64_t dd) { return grid_for(dd, 256 * 8, kMaxStatParts); }

cudaError_t launch_sumsq(const float* S, int batch, int64_t dd, float* part, int64_t part_ld, cudaStream_t st) {
  const int per_mat = sumsq_parts(dd);
  if (per_mat > part_ld) return cudaErrorInvalidValue;
  dim3 grid(per_mat, batch);
  k_sumsq<<<grid, 256, 0, st>>>(S, dd, part, part_ld);
  return cudaGetLastError();
}

cudaError_t launch_requant(const float* P, int batch, int d, __half* Ph, __half* PhT, __half* Pl, __half* PlT,
                           int64_t ld16, int64_t mat16, float* scal, int scal_ld, int slot, cudaStream_t st) {
  k_fill_scal<<<(batch + 127) / 128, 128, 0, st>>>(scal, scal_ld, slot, batch, 0.0f);
  const int64_t dd = static_cast<int64_t>(d) * d;
  dim3 g1(grid_for(dd, 256 * 8, 1024), batch);
  k_amax<<<g1, 256, 0, st>>>(P, dd, scal, scal_ld, slot);
  k_requant_scale<<<(batch + 127) / 128, 128, 0, st>>>(batch, scal, scal_ld, slot);
  dim3 grid((d + 31) / 32, (d + 31) / 32, batch), block(32, 8);
  k_requant<<<grid, block, 0, st>>>(P, d, Ph, PhT, Pl, PlT, ld16, mat16, scal, scal_ld, slot);
  return cudaGetLastError();
}

cudaError_t launch_reset_factor(float* S, float* P, __half* Ph, __half* PhT, __half* Pl, __half* PlT, int d,
                                int64_t ld16, int64_t mat16, int batch, float eps, float* scal, int scal_ld,
                                int pi_slot, cudaStream_t st) {
  const int64_t tot = static_cast<int64_t>(d) * d * batch;
  k_reset_factor<<<grid_for(tot, 256, 8192), 256, 0, st>>>(S, P, Ph, PhT, Pl, PlT, d, ld16, mat16, batch, eps);
  k_fill_scal<<<(batch + 127) / 128, 128, 0, st>>>(scal, scal_ld, pi_slot, batch,
                                                   ldexpf(1.0f, -kHeadroom));
  return cudaGetLastError();
}

}  // namespace okls

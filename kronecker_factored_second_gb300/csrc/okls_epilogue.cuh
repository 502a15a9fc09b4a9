// Tile decoding and the fused OKLS epilogues of the tcgen05 GEMM kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "okls_internal.h"

namespace okls {

struct TileCoord {
  int p, mat, tm, tn;
  int64_t lt;  // tile index within its matrix
};

// Tile t of the launch's linear tile space.  Output tiles are kBM x kBN
// (128 x 256); symmetric problems keep the tiles that touch the upper
// triangle: column block >= floor(tm * kBM / kBN).  `p` is the caller's
// running problem index: tiles are visited in increasing order, so the
// search only moves forward.
__device__ __forceinline__ TileCoord decode_tile(const GemmProblem* probs, int nprob, int64_t t, int& p) {
  constexpr int kDiv = kBN / kBM;
  TileCoord c;
  while (p + 1 < nprob && t >= probs[p + 1].tile_begin) ++p;
  const GemmProblem& P = probs[p];
  // tile indices of a launch stay below 2^31 (checked on the host), so the
  // divisions run in 32 bits by multiplication
  const uint32_t local = static_cast<uint32_t>(t - P.tile_begin);
  c.p = p;
  const uint32_t mat = fastdiv(local, P.tpm_mul, P.tpm_shift);
  c.mat = static_cast<int>(mat);
  uint32_t r = local - mat * static_cast<uint32_t>(P.tiles_per_mat);
  c.lt = r;
  if (P.sym) {
    int tm = 0;
    for (;;) {
      const uint32_t cnt = static_cast<uint32_t>(P.tiles_n - tm / kDiv);
      if (r < cnt) break;
      r -= cnt;
      ++tm;
    }
    c.tm = tm;
    c.tn = tm / kDiv + static_cast<int>(r);
  } else {
    const uint32_t g = fastdiv(r, P.span_mul, P.span_shift);
    const int first = static_cast<int>(g) * P.group_m;
    const uint32_t rr = r - g * static_cast<uint32_t>(P.group_m * P.tiles_n);
    if (P.tiles_m - first >= P.group_m) {
      const uint32_t col = fastdiv(rr, P.gm_mul, P.gm_shift);
      c.tm = first + static_cast<int>(rr - col * static_cast<uint32_t>(P.group_m));
      c.tn = static_cast<int>(col);
    } else {  // the last, shorter group of row blocks
      const uint32_t col = fastdiv(rr, P.lgm_mul, P.lgm_shift);
      c.tm = first + static_cast<int>(rr - col * static_cast<uint32_t>(P.last_gm));
      c.tn = static_cast<int>(col);
    }
  }
  return c;
}

// Every loop below runs over the 32 values with a compile-time index and a
// predicate for the ragged edge, so the values never leave registers.

__device__ __forceinline__ void store_half32_row(__half* dst, const float (&x)[32], int nvalid) {
  if (nvalid == 32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __align__(16) __half2 h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(x[q * 8 + 2 * e], x[q * 8 + 2 * e + 1]);
      *reinterpret_cast<uint4*>(dst + q * 8) = *reinterpret_cast<uint4*>(h);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < nvalid) dst[e] = __float2half_rn(x[e]);
  }
}

// Split x into binary16 hi + lo (lo = r16(x - hi)).
__device__ __forceinline__ void split_lo(const float (&x)[32], float (&lo)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) lo[e] = x[e] - __half2float(__float2half_rn(x[e]));
}

// Row-major and transposed binary16 stores of 32 values of row i, columns
// j0..j0+31 of a square (ld16-pitched) output.
__device__ __forceinline__ void store_both16(__half* row_base, __half* t_base, int64_t ld16, int i, int j0,
                                             int cols, const float (&x)[32]) {
  const int nvalid = min(32, cols - j0);
  if (nvalid <= 0) return;
  store_half32_row(row_base + static_cast<int64_t>(i) * ld16 + j0, x, nvalid);
  if (t_base != nullptr) {
    // thread i writes column i of rows j0..: consecutive lanes hit
    // consecutive addresses of one row of the transposed output
    __half* t = t_base + static_cast<int64_t>(j0) * ld16 + i;
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < nvalid) t[static_cast<int64_t>(e) * ld16] = __float2half_rn(x[e]);
  }
}

__device__ __forceinline__ void store_f32_row(float* dst, const float (&x)[32], float scale, int nvalid,
                                              bool vec_ok) {
  if (vec_ok && nvalid == 32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(dst + 4 * q) =
          make_float4(x[4 * q] * scale, x[4 * q + 1] * scale, x[4 * q + 2] * scale, x[4 * q + 3] * scale);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < nvalid) dst[e] = x[e] * scale;
  }
}

__device__ __forceinline__ float scal_at(const GemmProblem& P, int slot, int mat) {
  return P.scal[static_cast<int64_t>(slot) * P.scal_ld + mat];
}

// Epilogue for one 32-column chunk of one accumulator row.
__device__ __forceinline__ void epilogue_chunk(const GemmProblem& P, const TileCoord& tc, int i, int j0,
                                               float (&v)[32], uint32_t& flags, float& sumsq) {
  if (i >= P.rows || j0 >= P.cols) return;
  const int nvalid = min(32, P.cols - j0);
  switch (P.epi) {
    case EPI_X16: {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] *= P.alpha;
      __half* dst = reinterpret_cast<__half*>(P.out_hi) + static_cast<int64_t>(tc.mat) * P.mat16 +
                    static_cast<int64_t>(i) * P.ld16 + j0;
      store_half32_row(dst, v, nvalid);
      bool bad = false;
#pragma unroll
      for (int e = 0; e < 32; ++e) bad |= !isfinite(v[e]);
      if (bad && P.check_finite) flags |= kStNonfiniteIter;
      break;
    }
    case EPI_NS_T:
    case EPI_NS_SCALE:
    case EPI_NS_LAST: {
      if (P.epi == EPI_NS_LAST) {
        float* dst = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32 + static_cast<int64_t>(i) * P.ld32 + j0;
        store_f32_row(dst, v, scal_at(P, P.scal_slot, tc.mat), nvalid, (P.ld32 & 3) == 0);
      }
      if (P.epi == EPI_NS_T) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = fmaf(P.beta, v[e], (i == j0 + e) ? P.alpha : 0.0f);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= P.alpha;
      }
      bool bad = false;
#pragma unroll
      for (int e = 0; e < 32; ++e) bad |= !isfinite(v[e]) || fabsf(v[e]) > 65504.0f;
      if (bad) flags |= kStNonfiniteIter;
      const int64_t moff = static_cast<int64_t>(tc.mat) * P.mat16;
      __half* hi = reinterpret_cast<__half*>(P.out_hi) + moff;
      __half* hit = P.out_hi_t ? reinterpret_cast<__half*>(P.out_hi_t) + moff : nullptr;
      if (P.split_out) {
        float lo[32];
        split_lo(v, lo);
        store_both16(hi, hit, P.ld16, i, j0, P.cols, v);
        __half* lob = reinterpret_cast<__half*>(P.out_lo) + moff;
        __half* lot = P.out_lo_t ? reinterpret_cast<__half*>(P.out_lo_t) + moff : nullptr;
        store_both16(lob, lot, P.ld16, i, j0, P.cols, lo);
      } else {
        store_both16(hi, hit, P.ld16, i, j0, P.cols, v);
      }
      break;
    }
    case EPI_SYRK: {
      // S <- beta2 S + alpha acc + gamma I on and above the diagonal only; the
      // lower triangle is written later by the normaliser
      const float alpha = scal_at(P, P.scal_slot, tc.mat);
      float* S = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32 + static_cast<int64_t>(i) * P.ld32 + j0;
      if (j0 + 32 <= i) break;  // chunk entirely below the diagonal
      if (j0 >= i + 1 && nvalid == 32 && (P.ld32 & 3) == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 o = *reinterpret_cast<float4*>(S + 4 * q);
          o.x = fmaf(P.beta, o.x, alpha * v[4 * q + 0]);
          o.y = fmaf(P.beta, o.y, alpha * v[4 * q + 1]);
          o.z = fmaf(P.beta, o.z, alpha * v[4 * q + 2]);
          o.w = fmaf(P.beta, o.w, alpha * v[4 * q + 3]);
          *reinterpret_cast<float4*>(S + 4 * q) = o;
          sumsq += 2.0f * (o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = j0 + e;
          if (e < nvalid && j >= i) {
            float s = fmaf(P.beta, S[e], alpha * v[e]);
            if (j == i) s += P.gamma;
            S[e] = s;
            sumsq += (j == i ? 1.0f : 2.0f) * s * s;
          }
        }
      }
      break;
    }
    case EPI_UPDATE: {
      const float coef = P.beta * scal_at(P, P.scal_slot, tc.mat);
      const float decay = P.alpha;
      const int64_t off = static_cast<int64_t>(tc.mat) * P.mat32 + static_cast<int64_t>(i) * P.ld32 + j0;
      bool bad = false;
      if (P.w_bf16) {
        __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(P.w) + off;
        if (nvalid == 32 && (P.ld32 & 7) == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 raw = *reinterpret_cast<const uint4*>(w + 8 * q);
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 o = __bfloat1622float2(h[e]);
              const float n0 = fmaf(-coef, v[8 * q + 2 * e], decay * o.x);
              const float n1 = fmaf(-coef, v[8 * q + 2 * e + 1], decay * o.y);
              bad |= !isfinite(n0) || !isfinite(n1);
              h[e] = __floats2bfloat162_rn(n0, n1);
            }
            *reinterpret_cast<uint4*>(w + 8 * q) = raw;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e < nvalid) {
              const float nw = fmaf(-coef, v[e], decay * __bfloat162float(w[e]));
              bad |= !isfinite(nw);
              w[e] = __float2bfloat16_rn(nw);
            }
          }
        }
      } else {
        float* w = reinterpret_cast<float*>(P.w) + off;
        if (nvalid == 32 && (P.ld32 & 3) == 0) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 o = *reinterpret_cast<float4*>(w + 4 * q);
            o.x = fmaf(-coef, v[4 * q + 0], decay * o.x);
            o.y = fmaf(-coef, v[4 * q + 1], decay * o.y);
            o.z = fmaf(-coef, v[4 * q + 2], decay * o.z);
            o.w = fmaf(-coef, v[4 * q + 3], decay * o.w);
            bad |= !isfinite(o.x) || !isfinite(o.y) || !isfinite(o.z) || !isfinite(o.w);
            *reinterpret_cast<float4*>(w + 4 * q) = o;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e < nvalid) {
              const float nw = fmaf(-coef, v[e], decay * w[e]);
              bad |= !isfinite(nw);
              w[e] = nw;
            }
          }
        }
      }
      if (bad) flags |= kStNonfiniteUpdate;
      break;
    }
    case EPI_ROOT: {
      float* dst = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32 + static_cast<int64_t>(i) * P.ld32 + j0;
      store_f32_row(dst, v, scal_at(P, P.scal_slot, tc.mat), nvalid, (P.ld32 & 3) == 0);
      break;
    }
    default:
      break;
  }
}

}  // namespace okls

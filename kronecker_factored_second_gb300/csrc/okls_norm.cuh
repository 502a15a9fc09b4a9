// The first Newton-Schulz step of one element, shared by the normaliser
// kernel and the fused small-factor chain so both round identically:
//   Y_0 = (S + rho c I) / c'  (times the 2^h headroom),  T_0 = a_0 I + b_0 Y_0,
//   Z_1 = T_0 2^-z_1,
// each stored as binary16 (and a low half in the split mode).
#pragma once

#include <cuda_fp16.h>

namespace okls {

struct NormOut {
  __half y, t, z, yl, tl, zl;
  bool bad;
};

__device__ __forceinline__ NormOut norm_value_core(float s, bool diag, float inv, float rc, float a0h, float b0,
                                                  float zsc, bool split_y, bool split_t, bool split_z) {
  NormOut o;
  const float y = (s + (diag ? rc : 0.0f)) * inv;
  o.y = __float2half_rn(y);
  float yv = __half2float(o.y);
  o.yl = __float2half_rn(0.0f);
  if (split_y) {
    o.yl = __float2half_rn(y - yv);
    yv += __half2float(o.yl);
  }
  const float t = fmaf(b0, yv, diag ? a0h : 0.0f);
  o.t = __float2half_rn(t);
  float tv = __half2float(o.t);
  o.tl = __float2half_rn(0.0f);
  if (split_t) {
    o.tl = __float2half_rn(t - tv);
    tv += __half2float(o.tl);
  }
  const float z = tv * zsc;
  o.z = __float2half_rn(z);
  o.zl = split_z ? __float2half_rn(z - __half2float(o.z)) : __float2half_rn(0.0f);
  o.bad = !isfinite(y);
  return o;
}

}  // namespace okls

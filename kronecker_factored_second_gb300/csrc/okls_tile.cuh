// Small dense products staged in shared memory (fp32, CUDA cores), shared by
// the one-CTA kernels of the SOAP and Clean modes.
#pragma once

namespace okls {

// r x c = op(A) op(B) over K = k from shared memory; each thread forms 4 x 4
// outputs and hands each one to out(i, j, value).  Rows and columns past r,
// c read whatever the padded buffers hold and are discarded, so every buffer
// needs rows and columns up to the next multiple of 4 inside its allocation.
// ta: A is staged k x r; tb: B is staged c x k.  Odd pitches keep the rows a
// warp's tiles read at one k in distinct banks.
template <class F>
__device__ __forceinline__ void tile_mm4(const float* A, int lda, bool ta, const float* B, int ldb, bool tb, int r,
                                         int c, int k, F&& out) {
  const int tr = (r + 3) >> 2, tcn = (c + 3) >> 2;
  for (int blk = threadIdx.x; blk < tr * tcn; blk += blockDim.x) {
    const int i0 = (blk / tcn) << 2, j0 = (blk % tcn) << 2;
    float acc[4][4] = {};
    for (int q = 0; q < k; ++q) {
      float av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = ta ? A[q * lda + i0 + u] : A[(i0 + u) * lda + q];
        bv[u] = tb ? B[(j0 + u) * ldb + q] : B[q * ldb + j0 + u];
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

}  // namespace okls

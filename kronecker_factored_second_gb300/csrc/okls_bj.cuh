// The blocked Jacobi solver's layout and pairing (okls_bjacobi.cu; the
// tensor-core panel products of okls_tc3.cu read the same buffers).
#pragma once

#include <stdint.h>

#include "okls_internal.h"

namespace okls {
namespace bj {

constexpr int kB = 64;             // block edge
constexpr int kP = 2 * kB;         // pair subproblem edge
constexpr int kParts = 32;         // fixed-slot partial sums of the stopping rule

__host__ __device__ inline int64_t r4(int64_t x) { return (x + 3) & ~int64_t(3); }

// per-matrix scratch, in floats: A in the current round's layout and its
// image A P, the basis panels (two: they alternate round by round), the pair
// rotations, flags, the per-position arrays of the finish and the partials
struct Layout {
  int64_t kk, a0, a1, q0, q1, vv, vimg, flags, lam, inv, orig, sign, parts, misc, total;
};

// V^T of a pair as the tensor-core panel product's A operand: for each of the
// two 64-deep K-blocks the three bf16 terms, each a 128-row x 128-byte image
// in the 128-byte-swizzled K-major layout (16 KB): 96 KB per pair
constexpr int kVimgFloats = 2 * 3 * kP * 64 / 2;

__host__ __device__ inline Layout layout(int kp) {
  Layout L;
  const int64_t np = kp / kP;
  L.kk = static_cast<int64_t>(kp) * kp;
  L.a0 = 0;
  L.a1 = L.a0 + L.kk;
  L.q0 = L.a1 + L.kk;
  L.q1 = L.q0 + L.kk;
  L.vv = L.q1 + L.kk;
  L.vimg = L.vv + np * kP * kP;
  L.flags = L.vimg + np * kVimgFloats;
  L.lam = L.flags + r4(np);
  L.inv = L.lam + r4(kp);
  L.orig = L.inv + r4(kp);
  L.sign = L.orig + r4(kp);
  L.parts = L.sign + r4(kp);
  L.misc = L.parts + 4 * kParts;  // doubles: off, diag per part
  L.total = L.misc + 4;           // [0] done, [1] sweeps (ints), [2] d2 (float)
  return L;
}

inline int padded(int d) { return (d + kP - 1) / kP * kP; }

struct Args {
  const float* A;      // count x d x d
  const float* Qh;     // count x d x d
  const float* Qprev;  // count x d x d
  float* Qout;         // count x d x d (may be Qprev)
  float* scratch;      // count x layout(kp).total
  int d, kp, nb, count;
  float tol2;
  const uint32_t* status;
  uint32_t* status_w;
};

struct Mat {
  float *a0, *a1, *q0, *q1, *vv, *vimg, *lam, *sign;
  int *flags, *inv, *orig;
  double* parts;
  int* misc;
  float* d2;
};

__device__ __forceinline__ Mat mat(const Args& P, int b) {
  const Layout L = layout(P.kp);
  float* s = P.scratch + static_cast<int64_t>(b) * L.total;
  Mat M;
  M.a0 = s + L.a0;
  M.a1 = s + L.a1;
  M.q0 = s + L.q0;
  M.q1 = s + L.q1;
  M.vv = s + L.vv;
  M.vimg = s + L.vimg;
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

// the whole CTA leaves once the status word is set or the matrix is done
__device__ __forceinline__ bool skip(const Args& P, const Mat& M) {
  return __syncthreads_or(threadIdx.x == 0 &&
                          (*reinterpret_cast<const volatile uint32_t*>(P.status) != 0u ||
                           *reinterpret_cast<volatile int*>(M.misc) != 0));
}

// A panel product's source and destination buffers and how rows and columns
// move: out = V_q^T (src rows 128q..), or the rows themselves when pair q was
// not rotated, written to dst
//   mode 0: transposed, dst[c][128q + i]
//   mode 1: rows and columns moved to round rd + 1's block positions
//   mode 2: rows moved to round rd + 1's block positions
struct Panel {
  int src_buf, dst_buf, mode;  // buffers: 0 a0, 1 a1, 2 q0, 3 q1
};

__device__ __forceinline__ float* buf(const Mat& M, int i) {
  return i == 0 ? M.a0 : i == 1 ? M.a1 : i == 2 ? M.q0 : M.q1;
}

// destination of element (row, col) of the pair-q panel tile (row in 0..127,
// col an absolute column)
__device__ __forceinline__ int64_t panel_dst(int mode, int q, int row, int col, int rd, int nb, int kp) {
  if (mode == 0) return static_cast<int64_t>(col) * kp + q * kP + row;
  const int r = next_pos(2 * q + row / kB, rd, nb) * kB + (row & (kB - 1));
  const int c = mode == 1 ? next_pos(col / kB, rd, nb) * kB + (col & (kB - 1)) : col;
  return static_cast<int64_t>(r) * kp + c;
}

}  // namespace bj

// The tensor-core panel products of one round (okls_tc3.cu): the pair-q
// panels of t0 (and t1 when ntarget == 2) for every matrix.
cudaError_t launch_t3_panels(const bj::Args& P, int rd, bj::Panel t0, bj::Panel t1, int ntarget, cudaStream_t st);

}  // namespace okls

// Fused Newton-Schulz chain for small factors (d <= 128), one CTA per factor
// matrix, everything on chip (sm_103a).
//
// Page "Online KL Shampoo" (README, bullet list and "How it works"): the
// inverse root P = S^-1/2 by a 10-step scaled coupled Newton-Schulz
// iteration, 27 binary16 GEMMs with fp32 accumulation.  For d <= 128 a whole
// factor fits in one SM: Y_k, Z_k (two ping-pong copies each) and T_k are
// 128 x 128 binary16 tiles in shared memory, the products run as tcgen05.mma
// (M128 N128 K16) into Tensor Memory, and the epilogues write the next
// iterates straight back into shared memory.  One launch replaces the
// normaliser and the 19 GEMM launches of the general path; the arithmetic is
// the same: the same binary16 roundings, scales and coupled order
// (M_k = Z_k Y_k, Y_{k+1} = Y_k T_k, Z_{k+1} = T_k Z_k).
//
// Shared-memory layout of a 128 x 128 binary16 matrix X: two 64-column
// chunks of 128 rows x 128 bytes (16 KB each), rows 128-byte swizzled
// (16-byte unit u of row r stored at unit u ^ (r % 8)).  The same bytes are a
// K-major operand (A = X: 8-row groups 1024 B apart, K advanced inside the
// 128-byte row, next 64 K in the next chunk) and an MN-major operand
// (B = X as K x N: N chunks 16 KB apart, 8 K-rows 1024 B apart, K advanced by
// 16 rows = 2048 B), so no transposed copy is ever formed.
//
// Rows and columns beyond d stay zero: the identity terms are added on the
// valid diagonal only, so the padding never feeds the valid block.
#include <cuda_fp16.h>

#include "okls_internal.h"
#include "okls_kernels.h"
#include "okls_norm.cuh"
#include "okls_ptx.cuh"

namespace okls {

constexpr int kSD = 128;                  // padded factor edge
constexpr int kSChunk = kSD * 128;        // bytes of one 64-column chunk
constexpr int kSMat = 2 * kSChunk;        // bytes of one binary16 matrix
constexpr int kSmallThreads = 128;        // 4 warps: TMEM lane quarters
constexpr int kSmallSmem = 5 * kSMat + 1024 /*align*/ + 64 /*barrier, TMEM slot*/;

// byte offset of the 16-byte unit holding columns [col, col + 8) of row
__device__ __forceinline__ uint32_t sw_off(int row, int col) {
  return static_cast<uint32_t>((col >> 6) * kSChunk + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

// MN-major descriptor with an explicit leading-byte offset (N-chunk stride)
__device__ __forceinline__ uint64_t mn_desc_lbo(uint32_t saddr, uint32_t lbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// D (TMEM column offset dcol) = A * B for two resident 128 x 128 matrices
__device__ __forceinline__ void small_mma(uint32_t tmem, uint32_t dcol, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = idesc_f16_f32(kSD, kSD, true);
#pragma unroll
  for (int kk = 0; kk < kSD / kUmmaK; ++kk) {
    const uint64_t ad = sw128_desc(a + (kk >> 2) * kSChunk + (kk & 3) * 32);
    const uint64_t bd = mn_desc_lbo(b + kk * kUmmaK * 128, kSChunk);
    umma_f16(tmem + dcol, ad, bd, idesc, kk != 0 ? 1u : 0u);
  }
}

// 8 binary16 values of row `row`, columns [c, c+8): into shared memory
// (swizzled) and, when given, into a row-major global copy of the valid block
__device__ __forceinline__ void put8(uint8_t* sm, int row, int c, const __half (&h)[8], __half* g, int64_t ldg,
                                     int d) {
  *reinterpret_cast<uint4*>(sm + sw_off(row, c)) = *reinterpret_cast<const uint4*>(h);
  if (g && row < d) {
    if (c + 8 <= d && (ldg & 7) == 0) {
      *reinterpret_cast<uint4*>(g + static_cast<int64_t>(row) * ldg + c) = *reinterpret_cast<const uint4*>(h);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c + e < d) g[static_cast<int64_t>(row) * ldg + c + e] = h[e];
    }
  }
}

enum SmallEpi { SE_SCALE = 0, SE_T = 1, SE_LAST = 2, SE_ROOT = 3 };

// Epilogue of one accumulator: this thread's row, all 128 columns.
__device__ __forceinline__ void small_epilogue(uint32_t tmem, uint32_t dcol, int kind, uint8_t* dst, int row, int d,
                                               float alpha, float beta, __half* gcopy, int64_t ldg, float* g32,
                                               float scale32, uint32_t& flags) {
  const int warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int c = 0; c < kSD; c += 32) {
    float v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + dcol + c, v);
    if (kind == SE_LAST || kind == SE_ROOT) {
      if (row < d) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c + e < d) g32[static_cast<int64_t>(row) * d + c + e] = v[e] * scale32;
      }
      if (kind == SE_ROOT) continue;
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      if (kind == SE_T)
        v[e] = fmaf(beta, v[e], (row == c + e && row < d) ? alpha : 0.0f);
      else
        v[e] *= alpha;
      if (!isfinite(v[e]) || fabsf(v[e]) > 65504.0f) flags |= kStNonfiniteIter;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __align__(16) __half h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(v[q * 8 + e]);
      if (kind == SE_LAST) {
        // P^ goes to global memory only
        if (row < d) {
          const int cc = c + q * 8;
          if (cc + 8 <= d && (ldg & 7) == 0) {
            *reinterpret_cast<uint4*>(gcopy + static_cast<int64_t>(row) * ldg + cc) = *reinterpret_cast<const uint4*>(h);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (cc + e < d) gcopy[static_cast<int64_t>(row) * ldg + cc + e] = h[e];
          }
        }
      } else {
        put8(dst, row, c + q * 8, h, gcopy, ldg, d);
      }
    }
  }
}

// Generic-proxy writes to shared memory become visible to the tensor core,
// every thread's TMEM reads are ordered before the next MMA.
__device__ __forceinline__ void small_sync_for_mma() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__global__ void __launch_bounds__(kSmallThreads, 1) okls_ns_small_kernel(const __grid_constant__ SmallNsArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ys[2] = {smem, smem + kSMat};
  uint8_t* Zs[2] = {smem + 2 * kSMat, smem + 3 * kSMat};
  uint8_t* Ts = smem + 4 * kSMat;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 5 * kSMat);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  __shared__ int skip;

  const int tid = threadIdx.x;
  const int fi = blockIdx.x < A.f[0].count ? 0 : 1;
  const SmallNsFactor& F = A.f[fi];
  const int mat = fi == 0 ? blockIdx.x : blockIdx.x - A.f[0].count;
  const int d = F.d;
  const int row = tid;  // one accumulator lane (matrix row) per thread

  if (tid == 0) {
    skip = (*reinterpret_cast<volatile uint32_t*>(A.status) != 0u) ? 1 : 0;
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (skip) return;
  if ((tid >> 5) == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = A.iters;
  const int h = kHeadroom;
  auto slotv = [&](int slot) { return A.scal[static_cast<int64_t>(slot) * A.scal_ld + mat]; };
  uint16_t* trace = fi == 0 ? A.trace : nullptr;
  const int64_t tdd = static_cast<int64_t>(d) * d;
  auto trace_slice = [&](int k) -> __half* {
    return trace ? reinterpret_cast<__half*>(trace) + (static_cast<int64_t>(k) * A.trace_count + mat) * tdd : nullptr;
  };
  uint32_t flags = 0;

  // ---- normaliser: Y_0, T_0, Z_1 from the fp32 factor (one row per thread)
  {
    float* S = F.S + static_cast<int64_t>(mat) * d * d;
    const float cp = slotv(F.slot_cprime);
    const float c = sqrtf(slotv(F.slot_sumsq));
    const float inv = ldexpf(1.0f, h) / cp;
    const float rc = A.ridge * c;
    const float a0h = ldexpf(A.a[0], h);
    const float zsc = ldexpf(1.0f, -A.z[1]);
    __half* ty = trace_slice(0);
    __half* tz0 = trace_slice(1);
    __half* tt = trace_slice(2);
    bool bad = false;
#pragma unroll 1
    for (int c0 = 0; c0 < kSD; c0 += 8) {
      __align__(16) __half hy[8], ht[8], hz[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = c0 + e;
        float s = 0.0f;
        if (row < d && j < d) {
          if (F.upper_only)
            s = j >= row ? S[static_cast<int64_t>(row) * d + j] : S[static_cast<int64_t>(j) * d + row];
          else
            s = 0.5f * (S[static_cast<int64_t>(row) * d + j] + S[static_cast<int64_t>(j) * d + row]);
        }
        if (row < d && j < d) {
          const NormOut o = norm_value_core(s, row == j, inv, rc, a0h, A.b[0], zsc, false, false, false);
          hy[e] = o.y;
          ht[e] = o.t;
          hz[e] = o.z;
          bad |= o.bad;
        } else {
          hy[e] = ht[e] = hz[e] = __float2half_rn(0.0f);
        }
      }
      put8(Ys[0], row, c0, hy, ty, d, d);
      put8(Ts, row, c0, ht, tt, d, d);
      put8(Zs[1], row, c0, hz, nullptr, d, d);
      if (tz0 && row < d) {  // Z_0 = I is not stored: zeros, as the general path
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c0 + e < d) tz0[static_cast<int64_t>(row) * d + c0 + e] = __float2half_rn(0.0f);
      }
    }
    if (bad) flags |= kStNonfiniteIter;
    // the state keeps both triangles: the lower one mirrors the product's upper one
    __syncthreads();
    if (F.upper_only && row < d) {
      for (int j = 0; j < row; ++j) S[static_cast<int64_t>(row) * d + j] = S[static_cast<int64_t>(j) * d + row];
    }
  }

  uint32_t phase = 0;
  auto run = [&](void (*issue)(uint32_t, const uint8_t*, const uint8_t*, const uint8_t*, const uint8_t*),
                 const uint8_t* p0, const uint8_t* p1, const uint8_t* p2, const uint8_t* p3) {
    small_sync_for_mma();
    if (tid == 0) {
      issue(tmem, p0, p1, p2, p3);
      umma_commit(bar);
    }
    __syncwarp();
    const bool mine = mbar_wait(bar, phase, A.status);
    phase ^= 1u;
    // every thread takes the same branch afterwards (a wait that gave up in
    // one thread must stop all of them before the next barrier)
    const bool all = __syncthreads_and(mine) != 0;
    tc_fence_after();
    return all;
  };
  auto one = [](uint32_t tm, const uint8_t* a, const uint8_t* b, const uint8_t*, const uint8_t*) {
    small_mma(tm, 0, smem_u32(a), smem_u32(b));
  };
  auto two = [](uint32_t tm, const uint8_t* a0, const uint8_t* b0, const uint8_t* a1, const uint8_t* b1) {
    small_mma(tm, 0, smem_u32(a0), smem_u32(b0));
    small_mma(tm, kSD, smem_u32(a1), smem_u32(b1));
  };

  bool ok = true;
  // ---- k = 0: Y_1 = Y_0 T_0 (Z_1 = T_0 came from the normaliser)
  ok = run(one, Ys[0], Ts, nullptr, nullptr);
  if (ok)
    small_epilogue(tmem, 0, SE_SCALE, Ys[1], row, d, ldexpf(1.0f, -h), 0.0f, K > 1 ? trace_slice(3) : nullptr, d,
                   nullptr, 0.0f, flags);
  if (ok && trace && K > 1 && row < d) {
    // Z_1 for iteration 1's slot
    __half* tz = trace_slice(4);
    for (int c0 = 0; c0 < d; c0 += 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(Zs[1] + sw_off(row, c0));
      const __half* hh = reinterpret_cast<const __half*>(&u);
      for (int e = 0; e < 8 && c0 + e < d; ++e) tz[static_cast<int64_t>(row) * d + c0 + e] = hh[e];
    }
  }
  for (int k = 1; k < K && ok; ++k) {
    const int cur = k & 1, nxt = cur ^ 1;
    // T_k = a_k I + b_k Z_k Y_k
    ok = run(one, Zs[cur], Ys[cur], nullptr, nullptr);
    if (!ok) break;
    small_epilogue(tmem, 0, SE_T, Ts, row, d, ldexpf(A.a[k], h), ldexpf(A.b[k], A.z[k] - h), trace_slice(3 * k + 2),
                   d, nullptr, 0.0f, flags);
    if (k < K - 1) {
      ok = run(two, Ys[cur], Ts, Ts, Zs[cur]);
      if (!ok) break;
      small_epilogue(tmem, 0, SE_SCALE, Ys[nxt], row, d, ldexpf(1.0f, -h), 0.0f, trace_slice(3 * (k + 1)), d,
                     nullptr, 0.0f, flags);
      small_epilogue(tmem, kSD, SE_SCALE, Zs[nxt], row, d, ldexpf(1.0f, A.z[k] - A.z[k + 1] - h), 0.0f,
                     trace_slice(3 * (k + 1) + 1), d, nullptr, 0.0f, flags);
    } else {
      // last step: Z_K -> P (fp32) and P^ (binary16); Y_K -> the square root.
      // An iterate that overflowed anywhere in this matrix's chain leaves its
      // P, P^, pi and root as they were.  (Each matrix is decided on its own:
      // other matrices of the launch whose chains finished keep their new
      // roots, each with its own scale.)
      ok = run(two, Ys[cur], Ts, Ts, Zs[cur]);
      if (!ok) break;
      if (__syncthreads_or(flags != 0u)) break;
      if (F.root32)
        small_epilogue(tmem, 0, SE_ROOT, nullptr, row, d, 0.0f, 0.0f, nullptr, 0,
                       F.root32 + static_cast<int64_t>(mat) * d * d, slotv(F.slot_rscale), flags);
      if (A.want_p) {
        __half* ph = F.Ph + static_cast<int64_t>(mat) * F.ph_mat;
        small_epilogue(tmem, kSD, SE_LAST, nullptr, row, d, ldexpf(1.0f, A.z[k] - A.z[k + 1] - h), 0.0f, ph,
                       F.ph_ld, F.P32 + static_cast<int64_t>(mat) * d * d, slotv(F.slot_pscale), flags);
        if (trace && row < d) {
          __half* tp = trace_slice(3 * K);
          for (int j = 0; j < d; ++j) tp[static_cast<int64_t>(row) * d + j] = ph[static_cast<int64_t>(row) * F.ph_ld + j];
        }
        // the scale of P^ (P = pi P^), written with it
        if (tid == 0) {
          const double cp = static_cast<double>(slotv(F.slot_cprime));
          A.scal[static_cast<int64_t>(F.slot_pi) * A.scal_ld + mat] = static_cast<float>(ldexp(1.0 / sqrt(cp), A.z[K] - h));
        }
      }
    }
  }
  if (flags) atomicOr(A.status, flags);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((tid >> 5) == 0) tmem_dealloc(tmem, 256);
}

cudaError_t launch_ns_small(const SmallNsArgs& A, cudaStream_t st) {
  static PerDevice pd;
  const cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(okls_ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
  });
  if (e != cudaSuccess) return e;
  const int blocks = A.f[0].count + (A.nf > 1 ? A.f[1].count : 0);
  if (blocks <= 0) return cudaSuccess;
  okls_ns_small_kernel<<<blocks, kSmallThreads, kSmallSmem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace okls

// fp32-accurate products on the tensor cores (sm_103a): tcgen05.mma with
// bf16 operands, every fp32 operand split into three bf16 terms.
//
// The fp32 products of SOAP (Clean page, Appendix C, Algorithm 4: the
// rotations G' = Q_L^T G Q_R, M' = Q_L^T M Q_R, N = Q_L N' Q_R^T, the factor
// updates, the refresh's basis products) and of Clean past one CTA (Clean
// page, Algorithm 1 and Appendix A, Algorithm 3: the sketches, Gram products,
// rotations into the bases) need fp32 accuracy: the bases must stay
// orthonormal to ~1e-6 and the eigen-decompositions resolve gaps of 1e-3 of
// the spectrum.  A binary16 or bf16 product would not do; an fp32 product on
// the CUDA cores runs at ~1/50 of the tensor rate.
//
// The split: x = b1 + b2 + b3 with b1 = bf16(x), b2 = bf16(x - b1),
// b3 = bf16(x - b1 - b2) (round to nearest; each difference is exact in
// fp32), and the three terms hold x exactly (|b2| <= 2^-8 |x|,
// |b3| <= 2^-17 |x|: three 8-bit terms with signed rounding cover fp32's
// 24-bit significand).  A product of two split values keeps six terms,
//   b1 c1 + b1 c2 + b2 c1 + b1 c3 + b3 c1 + b2 c2
// (down to 2^-15 of the leading one), each product of two bf16 values exact
// in the fp32 accumulator; what is left out (b2 c3 + b3 c2 + b3 c3) is at
// most 2^-24 of |x c|, fp32's unit roundoff.  The accumulation is fp32 in
// TMEM, so the result carries the rounding of an fp32 product with K-deep
// sums.  A value that bf16 holds exactly (an identity rotation, a bf16
// gradient) has b2 = b3 = 0 and its products are exact: multiplying by the
// identity reproduces the other operand bit for bit.
//
// The kernel: one CTA per 128 x 128 output tile, K in stages of 64 (one
// 128-byte bf16 row per operand row, the SWIZZLE_128B K-major layout that
// tcgen05 reads), two stages of A1 A2 A3 B1 B2 B3 (96 KB each).  Warps 8-14
// load the fp32 (or bf16) operand tiles with plain coalesced loads -- any
// layout, transposed or not, ragged edges read as zero -- split them and
// store the three parts; warp 15 allocates the TMEM accumulators and one of its
// threads issues the 24 MMAs of a stage; warps 0-7 add each stage's partial
// products into registers and store the tile.  Every wait is bounded.
#include <cuda_bf16.h>

#include "okls_bj.cuh"
#include "okls_internal.h"
#include "okls_kernels.h"
#include "okls_ptx.cuh"

namespace okls {

namespace {

constexpr int kT3M = 128;                   // tile rows: A rows, TMEM lanes
constexpr int kT3N = 128;                   // tile columns: B rows, TMEM columns
constexpr int kT3K = 64;                    // K per stage: one 128-byte row of bf16
constexpr int kT3Part = kT3M * kT3K * 2;    // 16 KB: one bf16 term of one operand tile
constexpr int kT3StageBytes = 6 * kT3Part;  // A1 A2 A3 B1 B2 B3
constexpr int kT3Stages = 2;
constexpr int kT3Drain = 256;               // warps 0-7: the K-block partials into registers, then the store
constexpr int kT3Prod = 224;                // warps 8-14: loads and splits (16 warps in all: 128 registers each)
constexpr int kT3Threads = kT3Drain + kT3Prod + 32;  // warp 15: TMEM and the MMA issue
constexpr int kT3Cols = 512;                // TMEM: two buffers x (leading term, corrections) x 128 columns
constexpr int kT3Smem = kT3Stages * kT3StageBytes + 1024 + 128;

// tcgen05.mma kind::f16 with A and B bf16 (format 1 at bits 7-9 and 10-12),
// D fp32, both K-major
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape), and
// the wait for the load
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// the three bf16 terms of 8 values, stored as chunk kc of row r of the three
// parts (row r at r * 128 bytes, 16-byte chunk kc at (kc ^ (r % 8)) * 16);
// pairs go through the packed two-value conversion
__device__ __forceinline__ void t3_store(uint8_t* part0, int r, int kc, const float (&v)[8]) {
  uint32_t w1[4], w2[4], w3[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float x0 = v[2 * u], x1 = v[2 * u + 1];
    const __nv_bfloat162 a = __floats2bfloat162_rn(x0, x1);
    const float r0 = x0 - __low2float(a), r1 = x1 - __high2float(a);
    const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
    const __nv_bfloat162 c = __floats2bfloat162_rn(r0 - __low2float(b), r1 - __high2float(b));
    w1[u] = *reinterpret_cast<const uint32_t*>(&a);
    w2[u] = *reinterpret_cast<const uint32_t*>(&b);
    w3[u] = *reinterpret_cast<const uint32_t*>(&c);
  }
  const uint32_t off = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(kc) ^ (r & 7u)) << 4);
  *reinterpret_cast<uint4*>(part0 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *reinterpret_cast<uint4*>(part0 + kT3Part + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  *reinterpret_cast<uint4*>(part0 + 2 * kT3Part + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
}

// An operand tile source: element (r, k) of the tile (r from the tile's first
// row, k from 0) at p[r * ld + k] (kmajor) or p[k * ld + r]; rows and K
// bound the valid part (zero past it); vec: 16-byte loads are aligned.
struct T3Src {
  const void* p;
  int64_t ld;
  int rows, K;
  int kmajor, bf16, vec;
};

template <bool kBf16>
__device__ __forceinline__ float t3_ld(const void* p, int64_t i) {
  if constexpr (kBf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  else return __ldg(reinterpret_cast<const float*>(p) + i);
}

// 4 consecutive elements at element offset i (16-byte fp32 or 8-byte bf16 load)
template <bool kBf16>
__device__ __forceinline__ float4 t3_ld4(const void* p, int64_t i) {
  if constexpr (kBf16) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p) + i));
    return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u), __uint_as_float(q.y << 16),
                       __uint_as_float(q.y & 0xffff0000u));
  } else {
    return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i));
  }
}

constexpr int kT3KItems = (kT3M * 8 + kT3Prod - 1) / kT3Prod;        // K-contiguous: (row, chunk) items per thread
constexpr int kT3MItems = (kT3M / 4 * 8 + kT3Prod - 1) / kT3Prod;    // row-contiguous: (row quad, chunk) items

// all producer threads: the stage's tile of one operand, K columns k0..k0+63.
// Every load of the thread is issued before the first split, so a stage
// waits for memory once.  A whole tile in range with aligned rows takes the
// vector path without per-element checks.
template <bool kKmajor, bool kBf16>
__device__ __forceinline__ void t3_fill_t(const T3Src& s, int k0, uint8_t* part0) {
  const int tid = threadIdx.x - kT3Drain;
  const bool whole = s.vec && s.rows >= kT3M && k0 + kT3K <= s.K;
  if constexpr (kKmajor) {
    // item (row r, chunk kc): 8 consecutive k of one row; 8 lanes per row
    float v[kT3KItems][8];
#pragma unroll
    for (int it = 0; it < kT3KItems; ++it) {
      const int idx = tid + it * kT3Prod;
      const int r = idx >> 3, k = k0 + 8 * (idx & 7);
      const int64_t o = static_cast<int64_t>(r) * s.ld + k;
      if (idx < kT3M * 8 && (whole || (s.vec && r < s.rows && k + 8 <= s.K))) {
        const float4 a = t3_ld4<kBf16>(s.p, o), b = t3_ld4<kBf16>(s.p, o + 4);
        v[it][0] = a.x; v[it][1] = a.y; v[it][2] = a.z; v[it][3] = a.w;
        v[it][4] = b.x; v[it][5] = b.y; v[it][6] = b.z; v[it][7] = b.w;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[it][u] = (idx < kT3M * 8 && r < s.rows && k + u < s.K) ? t3_ld<kBf16>(s.p, o + u) : 0.0f;
      }
    }
#pragma unroll
    for (int it = 0; it < kT3KItems; ++it) {
      const int idx = tid + it * kT3Prod;
      if (idx < kT3M * 8) t3_store(part0, idx >> 3, idx & 7, v[it]);
    }
  } else {
    // item (row quad rq, chunk kc): rows 4 rq .. 4 rq + 3 at the 8 k of chunk
    // kc, one 4-wide load per k; lanes run over kc first, so each store
    // instruction writes four whole 128-byte rows
    float v[kT3MItems][32];
#pragma unroll
    for (int it = 0; it < kT3MItems; ++it) {
      const int idx = tid + it * kT3Prod;
      const int kc = idx & 7, r = 4 * (idx >> 3);
      const int64_t o0 = static_cast<int64_t>(k0 + 8 * kc) * s.ld + r;
      if (idx < kT3M * 2 && whole) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 a = t3_ld4<kBf16>(s.p, o0 + u * s.ld);
          v[it][4 * u] = a.x;
          v[it][4 * u + 1] = a.y;
          v[it][4 * u + 2] = a.z;
          v[it][4 * u + 3] = a.w;
        }
      } else {
        const bool quad = idx < kT3M * 2 && r + 4 <= s.rows && s.vec;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = k0 + 8 * kc + u;
          const int64_t o = o0 + u * s.ld;
          if (quad) {
            const float4 a = k < s.K ? t3_ld4<kBf16>(s.p, o) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[it][4 * u] = a.x;
            v[it][4 * u + 1] = a.y;
            v[it][4 * u + 2] = a.z;
            v[it][4 * u + 3] = a.w;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              v[it][4 * u + i] = (idx < kT3M * 2 && r + i < s.rows && k < s.K) ? t3_ld<kBf16>(s.p, o + i) : 0.0f;
          }
        }
      }
    }
#pragma unroll
    for (int it = 0; it < kT3MItems; ++it) {
      const int idx = tid + it * kT3Prod;
      if (idx >= kT3M * 2) continue;
      const int kc = idx & 7, r = 4 * (idx >> 3);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = v[it][4 * u + i];
        t3_store(part0, r + i, kc, w);
      }
    }
  }
}

// the operand's layout and element type are uniform over the grid: one
// specialised fill per combination
__device__ __forceinline__ void t3_fill(const T3Src& s, int k0, uint8_t* part0) {
  if (s.kmajor) {
    if (s.bf16) t3_fill_t<true, true>(s, k0, part0);
    else t3_fill_t<true, false>(s, k0, part0);
  } else {
    if (s.bf16) t3_fill_t<false, true>(s, k0, part0);
    else t3_fill_t<false, false>(s, k0, part0);
  }
}

// A bounded wait that sleeps between tries: for the threads whose waits are
// not on the critical path (the drain warps, the producers when ahead), so
// that their polling does not take issue slots from the producers' splits.
__device__ __forceinline__ bool t3_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (ns < 256) ns *= 2;
    if (*reinterpret_cast<volatile uint32_t*>(status) & kStTimeout) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      atomicOr(status, kStTimeout);
      return false;
    }
  }
}

struct T3Smem {
  uint8_t* stage;  // kT3Stages x kT3StageBytes, 1024-byte aligned
  uint64_t* full;  // [stage] operands written (producers)
  uint64_t* empty; // [stage] operands read (MMA commit)
  uint64_t* accf;  // [buffer] K-block partial ready (MMA commit)
  uint64_t* acce;  // [buffer] partial drained (drain threads)
  uint64_t* fin;   // every MMA finished
  uint32_t* slot;
};

__device__ __forceinline__ T3Smem t3_smem(uint8_t* raw) {
  T3Smem S;
  const uintptr_t a = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
  S.stage = reinterpret_cast<uint8_t*>(a);
  uint64_t* bars = reinterpret_cast<uint64_t*>(S.stage + kT3Stages * kT3StageBytes);
  S.full = bars;
  S.empty = bars + 2;
  S.accf = bars + 4;
  S.acce = bars + 6;
  S.fin = bars + 8;
  S.slot = reinterpret_cast<uint32_t*>(bars + 9);
  return S;
}

// The pipeline of one output tile: fill(kb, A part 0, B part 0) by the
// producers; one thread issues each K-block's MMAs into a fresh pair of
// accumulators (the leading term b1 c1 and the five corrections) in one of
// two TMEM buffers; warps 0-7 add every K-block's pair into fp32 registers
// (round to nearest), so that no TMEM accumulator takes more than four MMAs
// of the leading term -- the tensor pipe's accumulation is not rounded to
// nearest, and over hundreds of MMAs its error would add up one way.  Then
// store(row, col0, v[32]) for the rows of each warp's TMEM lane quarter.
template <class Fill, class Store>
__device__ __forceinline__ void t3_tile(uint8_t* raw, int nkb, uint32_t* status, Fill fill, Store store) {
  const T3Smem S = t3_smem(raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kMmaWarp = (kT3Drain + kT3Prod) / 32;
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], kT3Prod);
      mbar_init(&S.empty[s], 1);
      mbar_init(&S.accf[s], 1);
      mbar_init(&S.acce[s], kT3Drain);
    }
    mbar_init(S.fin, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(S.slot, kT3Cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *S.slot;
  if (tid < kT3Drain) {
    // warp w: lanes of quarter w % 4 (tile rows), columns 64 (w / 4) ..
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float s0[32], s1[32];  // columns 64 h + 0..31 and 64 h + 32..63
#pragma unroll
    for (int i = 0; i < 32; ++i) s0[i] = s1[i] = 0.0f;
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int p = kb & 1;
      ok = t3_wait_sleep(&S.accf[p], (kb >> 1) & 1, status);
      tc_fence_after();
      if (ok) {
        const uint32_t col = lane_base + static_cast<uint32_t>(256 * p + 64 * h);
        float t[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* acc = c < 2 ? s0 + 16 * c : s1 + 16 * (c - 2);
          tmem_ld16(tmem + col + 128u + 16u * c, t);  // corrections
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] += t[i];
          tmem_ld16(tmem + col + 16u * c, t);         // leading term
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] += t[i];
        }
      }
      tc_fence_before();
      mbar_arrive(&S.acce[p]);
    }
    // a pipeline that gave up leaves no tile to store
    ok = ok && (*reinterpret_cast<volatile uint32_t*>(status) & kStTimeout) == 0u;
    if (ok) {
      store(32 * q + lane, 64 * h, s0);
      store(32 * q + lane, 64 * h + 32, s1);
    }
  } else if (tid < kT3Drain + kT3Prod) {
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb & 1;
      if (kb >= kT3Stages && !t3_wait_sleep(&S.empty[s], ((kb >> 1) - 1) & 1, status)) break;
      uint8_t* st = S.stage + s * kT3StageBytes;
      fill(kb, st, st + 3 * kT3Part);
      fence_proxy_async_shared();
      mbar_arrive(&S.full[s]);
    }
  } else if (lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(kT3M, kT3N);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb & 1, p = kb & 1;
      if (!mbar_wait(&S.full[s], (kb >> 1) & 1, status)) break;
      if (kb >= 2 && !mbar_wait(&S.acce[p], ((kb >> 1) - 1) & 1, status)) break;
      tc_fence_after();
      const uint32_t base = smem_u32(S.stage + s * kT3StageBytes);
      const uint64_t a1 = sw128_desc(base), a2 = sw128_desc(base + kT3Part), a3 = sw128_desc(base + 2 * kT3Part);
      const uint64_t b1 = sw128_desc(base + 3 * kT3Part), b2 = sw128_desc(base + 4 * kT3Part),
                     b3 = sw128_desc(base + 5 * kT3Part);
      const uint32_t d1 = tmem + static_cast<uint32_t>(256 * p), d2 = d1 + 128u;
#pragma unroll
      for (int k16 = 0; k16 < kT3K / 16; ++k16) {
        const uint64_t o = 2u * static_cast<uint32_t>(k16);  // 32 bytes in the 16-byte address field
        const uint32_t acc = k16 != 0 ? 1u : 0u;
        umma_f16(d1, a1 + o, b1 + o, idesc, acc);
        umma_f16(d2, a1 + o, b2 + o, idesc, acc);
        umma_f16(d2, a2 + o, b1 + o, idesc, 1u);
        umma_f16(d2, a1 + o, b3 + o, idesc, 1u);
        umma_f16(d2, a3 + o, b1 + o, idesc, 1u);
        umma_f16(d2, a2 + o, b2 + o, idesc, 1u);
      }
      umma_commit(&S.empty[s]);
      umma_commit(&S.accf[p]);
    }
    umma_commit(S.fin);
    // this thread's MMAs finish before the CTA may free the accumulators
    mbar_wait_own(S.fin, 0, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kT3Cols);
  }
}

__device__ __forceinline__ bool t3_flagged(const uint32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<const volatile uint32_t*>(status) != 0u);
}

// ---------------------------------------------------------------- the GEMM
// C[b] = alpha op(A[b]) op(B[b]) + beta_b C[b], the contract of k_cl_gemm.
__global__ void __launch_bounds__(kT3Threads, 1) k_t3_gemm(const __grid_constant__ ClGemm g) {
  extern __shared__ uint8_t t3_raw[];
  // like k_cl_gemm: skipped only when the caller guards the launch (the
  // status word itself only receives this kernel's timeouts)
  if (g.status_guard && t3_flagged(g.status_guard)) return;
  const int b = blockIdx.z;
  const int m0 = blockIdx.y * kT3M, n0 = blockIdx.x * kT3N;
  const size_t ea = g.a_bf16 ? 2 : 4, eb = g.b_bf16 ? 2 : 4;
  // A: element (r, k) of op(A) from row m0; B: element (n, k) of op(B)^T from row n0
  T3Src sa, sb;
  {
    const char* base = static_cast<const char*>(g.A) + static_cast<int64_t>(b) * g.sA * ea;
    sa.kmajor = g.ta ? 0 : 1;
    sa.p = base + (g.ta ? static_cast<int64_t>(m0) : static_cast<int64_t>(m0) * g.lda) * ea;
    sa.ld = g.lda;
    sa.rows = g.M - m0;
    sa.K = g.K;
    sa.bf16 = g.a_bf16;
    sa.vec = g.a_vec;
  }
  {
    const char* base = static_cast<const char*>(g.B) + static_cast<int64_t>(b) * g.sB * eb;
    sb.kmajor = g.tb ? 1 : 0;
    sb.p = base + (g.tb ? static_cast<int64_t>(n0) * g.ldb : static_cast<int64_t>(n0)) * eb;
    sb.ld = g.ldb;
    sb.rows = g.N - n0;
    sb.K = g.K;
    sb.bf16 = g.b_bf16;
    sb.vec = g.b_vec;
  }
  const float beta = g.beta_dev ? g.beta_dev[b] : g.beta;
  float* C = g.C + static_cast<int64_t>(b) * g.sC;
  const bool cvec = (g.ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
  const int nkb = (g.K + kT3K - 1) / kT3K;
  t3_tile(
      t3_raw, nkb, g.status,
      [&](int kb, uint8_t* pa, uint8_t* pb) {
        t3_fill(sa, kb * kT3K, pa);
        t3_fill(sb, kb * kT3K, pb);
      },
      [&](int r, int c0, const float (&v)[32]) {
        const int row = m0 + r;
        if (row >= g.M) return;
        float* out = C + static_cast<int64_t>(row) * g.ldc + n0 + c0;
        const int nc = min(32, g.N - n0 - c0);
        if (nc == 32 && cvec) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float4 o = make_float4(g.alpha * v[4 * u], g.alpha * v[4 * u + 1], g.alpha * v[4 * u + 2],
                                   g.alpha * v[4 * u + 3]);
            if (beta != 0.0f) {
              const float4 c = reinterpret_cast<const float4*>(out)[u];
              o.x = fmaf(beta, c.x, o.x);
              o.y = fmaf(beta, c.y, o.y);
              o.z = fmaf(beta, c.z, o.z);
              o.w = fmaf(beta, c.w, o.w);
            }
            reinterpret_cast<float4*>(out)[u] = o;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            if (u < nc) {
              float o = g.alpha * v[u];
              if (beta != 0.0f) o = fmaf(beta, out[u], o);
              out[u] = o;
            }
          }
        }
      });
}

// ------------------------------------------------- blocked Jacobi panels
// One CTA per (128-column tile, pair q, matrix x target): out (128 x 128) =
// V_q^T (src rows 128q.., the tile's columns), K = 128, written by the
// target's mode (okls_bj.cuh); a pair that was not rotated is copied (the
// transposing copy through shared memory).
__global__ void __launch_bounds__(kT3Threads, 1) k_t3_panel(const __grid_constant__ bj::Args P, int rd,
                                                           bj::Panel t0, bj::Panel t1, int ntarget) {
  extern __shared__ uint8_t t3_raw[];
  const int b = blockIdx.z / ntarget, which = blockIdx.z % ntarget;
  const bj::Panel T = which == 0 ? t0 : t1;
  const int q = blockIdx.y, c0 = blockIdx.x * kT3N;
  const bj::Mat M = bj::mat(P, b);
  if (bj::skip(P, M)) return;
  const int kp = P.kp, nb = P.nb;
  const float* src = bj::buf(M, T.src_buf) + static_cast<int64_t>(q) * bj::kP * kp + c0;
  float* dst = bj::buf(M, T.dst_buf);
  if (M.flags[q] == 0) {
    const int tid = threadIdx.x;
    if (T.mode == 0) {
      float* tile = reinterpret_cast<float*>(t3_raw);  // [i][c], pitch 129
      for (int e = tid; e < bj::kP * kT3N; e += kT3Threads) {
        const int i = e / kT3N, c = e % kT3N;
        tile[i * (kT3N + 1) + c] = src[static_cast<int64_t>(i) * kp + c];
      }
      __syncthreads();
      for (int e = tid; e < bj::kP * kT3N; e += kT3Threads) {
        const int c = e / bj::kP, i = e % bj::kP;
        dst[bj::panel_dst(0, q, i, c0 + c, rd, nb, kp)] = tile[i * (kT3N + 1) + c];
      }
    } else {
      for (int e = tid; e < bj::kP * kT3N; e += kT3Threads) {
        const int i = e / kT3N, c = e % kT3N;
        dst[bj::panel_dst(T.mode, q, i, c0 + c, rd, nb, kp)] = src[static_cast<int64_t>(i) * kp + c];
      }
    }
    return;
  }
  // A: V_q^T, split once by the solve kernel into the three terms' images
  const uint4* vimg = reinterpret_cast<const uint4*>(M.vimg + static_cast<int64_t>(q) * bj::kVimgFloats);
  T3Src sb;
  sb.p = src;  // element (c, l) at src[l][c]
  sb.ld = kp;
  sb.rows = kT3N;
  sb.K = bj::kP;
  sb.kmajor = 0;
  sb.bf16 = 0;
  sb.vec = 1;
  t3_tile(
      t3_raw, bj::kP / kT3K, P.status_w,
      [&](int kb, uint8_t* pa, uint8_t* pb) {
        const uint4* in = vimg + kb * (3 * kT3Part / 16);
        uint4* out = reinterpret_cast<uint4*>(pa);
        for (int i = threadIdx.x - kT3Drain; i < 3 * kT3Part / 16; i += kT3Prod) out[i] = __ldg(in + i);
        t3_fill(sb, kb * kT3K, pb);
      },
      [&](int r, int cl, const float (&v)[32]) {
        if (T.mode == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[bj::panel_dst(0, q, r, c0 + cl + j, rd, nb, kp)] = v[j];
        } else {
          // 32 consecutive columns inside one 64-column block
          float4* out = reinterpret_cast<float4*>(dst + bj::panel_dst(T.mode, q, r, c0 + cl, rd, nb, kp));
#pragma unroll
          for (int u = 0; u < 8; ++u) out[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
      });
}

}  // namespace

cudaError_t launch_t3_panels(const bj::Args& P, int rd, bj::Panel t0, bj::Panel t1, int ntarget, cudaStream_t st) {
  static PerDevice pd;
  cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(k_t3_panel, cudaFuncAttributeMaxDynamicSharedMemorySize, kT3Smem);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(P.kp / kT3N), static_cast<unsigned>(P.nb / 2),
                  static_cast<unsigned>(P.count * ntarget));
  k_t3_panel<<<grid, kT3Threads, kT3Smem, st>>>(P, rd, t0, t1, ntarget);
  return cudaGetLastError();
}

bool t3_gemm_eligible(const ClGemm& g) {
  if (!g.status) return false;
  static const int enabled = [] {
    const char* e = getenv("OKLS_TC3");
    return (e && e[0] == '0') ? 0 : 1;
  }();
  // the tensor-core path pays off once a tile has a few stages of K to run
  return enabled && g.M >= 64 && g.N >= 64 && g.K >= 128;
}

cudaError_t launch_t3_gemm(const ClGemm& g, cudaStream_t st) {
  static PerDevice pd;
  cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(k_t3_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kT3Smem);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((g.N + kT3N - 1) / kT3N, (g.M + kT3M - 1) / kT3M, g.batch);
  k_t3_gemm<<<grid, kT3Threads, kT3Smem, st>>>(g);
  return cudaGetLastError();
}

}  // namespace okls

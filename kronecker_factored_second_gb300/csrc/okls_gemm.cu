// Persistent tcgen05 GEMM with fused OKLS epilogues (sm_103a).
//
// One launch runs up to kMaxProblems independent batched problems
//   D[b] = sum_seg A_seg[b] * B_seg[b]^T      (A: rows x K, B: cols x K, both
//                                            K-contiguous binary16, fp32 acc)
// over one linear tile space.  Each CTA (one per SM) loops over tiles with a
// static stride; inside a CTA:
//   warp 0 / lane 0  TMA producer: 128x64 A and 256x64 B boxes, 128-byte
//                    swizzle, into a kStages-deep shared-memory ring;
//   warp 1 / lane 0  MMA issuer: four tcgen05.mma (M128 N256 K16) per stage
//                    into one of two 256-column TMEM accumulators;
//   warps 2-5        epilogue: tcgen05.ld of their 32 TMEM lanes, the fused
//                    OKLS arithmetic, global stores.
// The two accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.  All waits are bounded (okls_ptx.cuh).
//
// Where each epilogue comes from (page "Online KL Shampoo", "How it works"):
//   EPI_SYRK      the factor EMAs S <- beta2 S + (1-beta2)/n X X^T (+ eps I)
//   EPI_NS_T/SCALE/LAST  the coupled Newton-Schulz products of the inverse
//                 root (10 steps, 27 binary16 GEMMs, fp32 accumulation)
//   EPI_X16       the products G P_b, G^T P_a^T and P_a N feeding them
//   EPI_UPDATE    U = P_a N P_b and W <- W - lr wd (lr/lr_peak) W - lr c U
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "okls_internal.h"
#include "okls_ptx.cuh"

namespace okls {

struct TileCoord {
  int p, mat, tm, tn;
  int64_t lt;  // tile index within its matrix
};

__device__ __forceinline__ TileCoord decode_tile(const GemmLaunch& L, int64_t t) {
  TileCoord c;
  int p = 0;
  while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
  const GemmProblem& P = L.prob[p];
  const int64_t local = t - P.tile_begin;
  c.p = p;
  c.mat = static_cast<int>(local / P.tiles_per_mat);
  int64_t r = local - static_cast<int64_t>(c.mat) * P.tiles_per_mat;
  c.lt = r;
  if (P.sym) {
    // row block tm holds col blocks floor(tm/2) .. tiles_n-1 (BN = 2 BM)
    int tm = 0;
    for (;;) {
      const int cnt = P.tiles_n - tm / 2;
      if (r < cnt) break;
      r -= cnt;
      ++tm;
    }
    c.tm = tm;
    c.tn = tm / 2 + static_cast<int>(r);
  } else {
    const int64_t span = static_cast<int64_t>(kGroupM) * P.tiles_n;
    const int g = static_cast<int>(r / span);
    const int first = g * kGroupM;
    const int gm = min(kGroupM, P.tiles_m - first);
    const int64_t rr = r - static_cast<int64_t>(g) * span;
    c.tm = first + static_cast<int>(rr % gm);
    c.tn = static_cast<int>(rr / gm);
  }
  return c;
}

__device__ __forceinline__ void store_half32_row(__half* dst, const float (&x)[32], int nvalid,
                                                 bool vec_ok) {
  if (vec_ok && nvalid == 32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __align__(16) __half2 h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        h[e] = __floats2half2_rn(x[q * 8 + 2 * e], x[q * 8 + 2 * e + 1]);
      *reinterpret_cast<uint4*>(dst + q * 8) = *reinterpret_cast<uint4*>(h);
    }
  } else {
    for (int e = 0; e < nvalid; ++e) dst[e] = __float2half_rn(x[e]);
  }
}

// Split x into binary16 hi + lo (lo = r16(x - hi)).
__device__ __forceinline__ void split_lo(const float (&x)[32], float (&lo)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) lo[e] = x[e] - __half2float(__float2half_rn(x[e]));
}

// Row-major and transposed binary16 stores of 32 values of row i, columns
// j0..j0+31 of a square (ld16-pitched) output.
__device__ __forceinline__ void store_both16(__half* row_base, __half* t_base, int64_t ld16,
                                             int i, int j0, int cols, const float (&x)[32],
                                             bool vec_ok) {
  const int nvalid = min(32, cols - j0);
  if (nvalid <= 0) return;
  store_half32_row(row_base + static_cast<int64_t>(i) * ld16 + j0, x, nvalid, vec_ok);
  if (t_base != nullptr) {
    // thread i writes column i of rows j0..: consecutive lanes hit
    // consecutive addresses of one row of the transposed output
#pragma unroll 8
    for (int e = 0; e < nvalid; ++e)
      t_base[static_cast<int64_t>(j0 + e) * ld16 + i] = __float2half_rn(x[e]);
  }
}

__device__ __forceinline__ float scal_at(const GemmProblem& P, int slot, int mat) {
  return P.scal[static_cast<int64_t>(slot) * P.scal_ld + mat];
}

// Epilogue for one 32-column chunk of one accumulator row.
__device__ __forceinline__ void epilogue_chunk(const GemmProblem& P, const TileCoord& tc,
                                               int i, int j0, float (&v)[32], uint32_t& flags,
                                               float& sumsq) {
  if (i >= P.rows || j0 >= P.cols) return;
  const int nvalid = min(32, P.cols - j0);
  switch (P.epi) {
    case EPI_X16: {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] *= P.alpha;
      __half* dst = reinterpret_cast<__half*>(P.out_hi) + static_cast<int64_t>(tc.mat) * P.mat16 +
                    static_cast<int64_t>(i) * P.ld16 + j0;
      store_half32_row(dst, v, nvalid, true);
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
        const float ps = scal_at(P, P.scal_slot, tc.mat);
        float* dst = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32 +
                     static_cast<int64_t>(i) * P.ld32 + j0;
        const bool vec = (P.ld32 % 4 == 0) && nvalid == 32;
        if (vec) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 4 * q) =
                make_float4(v[4 * q] * ps, v[4 * q + 1] * ps, v[4 * q + 2] * ps, v[4 * q + 3] * ps);
        } else {
          for (int e = 0; e < nvalid; ++e) dst[e] = v[e] * ps;
        }
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
        store_both16(hi, hit, P.ld16, i, j0, P.cols, v, true);
        __half* lob = reinterpret_cast<__half*>(P.out_lo) + moff;
        __half* lot = P.out_lo_t ? reinterpret_cast<__half*>(P.out_lo_t) + moff : nullptr;
        store_both16(lob, lot, P.ld16, i, j0, P.cols, lo, true);
      } else {
        store_both16(hi, hit, P.ld16, i, j0, P.cols, v, true);
      }
      break;
    }
    case EPI_SYRK: {
      // only elements on or above the diagonal; mirrored below
      const float alpha = scal_at(P, P.scal_slot, tc.mat);
      float* S = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32;
      for (int e = 0; e < nvalid; ++e) {
        const int j = j0 + e;
        if (j < i) continue;
        const int64_t a = static_cast<int64_t>(i) * P.ld32 + j;
        float s = fmaf(P.beta, S[a], alpha * v[e]);
        if (j == i) s += P.gamma;
        S[a] = s;
        if (j != i) S[static_cast<int64_t>(j) * P.ld32 + i] = s;
        sumsq += (j == i ? 1.0f : 2.0f) * s * s;
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
        for (int e = 0; e < nvalid; ++e) {
          const float nw = fmaf(-coef, v[e], decay * __bfloat162float(w[e]));
          bad |= !isfinite(nw);
          w[e] = __float2bfloat16_rn(nw);
        }
      } else {
        float* w = reinterpret_cast<float*>(P.w) + off;
        const bool vec = (P.ld32 % 4 == 0) && nvalid == 32;
        if (vec) {
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
          for (int e = 0; e < nvalid; ++e) {
            const float nw = fmaf(-coef, v[e], decay * w[e]);
            bad |= !isfinite(nw);
            w[e] = nw;
          }
        }
      }
      if (bad) flags |= kStNonfiniteUpdate;
      break;
    }
    case EPI_ROOT: {
      const float rs = scal_at(P, P.scal_slot, tc.mat);
      float* dst = P.out32 + static_cast<int64_t>(tc.mat) * P.mat32 + static_cast<int64_t>(i) * P.ld32 + j0;
      for (int e = 0; e < nvalid; ++e) dst[e] = v[e] * rs;
      break;
    }
    default:
      break;
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) okls_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* skip = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // An earlier stage of the step failed: leave W, S and P untouched.
  if (threadIdx.x == 0) *skip = (*reinterpret_cast<volatile uint32_t*>(L.status) != 0u);
  __syncthreads();
  if (*skip) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      for (int p = 0; p < L.nprob; ++p)
        for (int s = 0; s < L.prob[p].nseg; ++s) {
          prefetch_tmap(L.maps + L.prob[p].amap[s]);
          prefetch_tmap(L.maps + L.prob[p].bmap[s]);
        }
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < L.total_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(L, t);
        const GemmProblem& P = L.prob[tc.p];
        const int nkb = (P.K + kBK - 1) / kBK;
        for (int sg = 0; sg < P.nseg && ok; ++sg) {
          const CUtensorMap* am = L.maps + P.amap[sg];
          const CUtensorMap* bm = L.maps + P.bmap[sg];
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, L.status)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * kStageBytes;
            uint8_t* sb = sa + kStageABytes;
            mbar_expect_tx(&full[stage], kStageBytes);
            tma_load_3d(sa, am, &full[stage], kb * kBK, tc.tm * kBM, tc.mat);
            tma_load_3d(sb, bm, &full[stage], kb * kBK, tc.tn * kBN, tc.mat);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // make sure no bulk copy is still landing in shared memory at exit
      const int64_t back = issued < kStages ? issued : kStages;
      for (int64_t q = 1; q <= back; ++q) {
        const int64_t idx = issued - q;
        const uint32_t s = static_cast<uint32_t>(idx % kStages);
        const uint32_t ph = static_cast<uint32_t>((idx / kStages) & 1);
        if (!mbar_wait(&full[s], ph, L.status)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_f16_f32(kBM, kBN);
      uint32_t stage = 0, phase = 0, it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < L.total_tiles && ok; t += gridDim.x, ++it) {
        const TileCoord tc = decode_tile(L, t);
        const GemmProblem& P = L.prob[tc.p];
        const int nkb = ((P.K + kBK - 1) / kBK) * P.nseg;
        const uint32_t buf = it & 1u;
        const uint32_t aph = (it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, L.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, L.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
          const uint32_t b0 = a0 + kStageABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            umma_f16(d, sw128_desc(a0 + kk * kUmmaK * 2), sw128_desc(b0 + kk * kUmmaK * 2), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      // all MMAs retired before TMEM is released
      umma_commit(drain);
      mbar_wait(drain, 0, L.status);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- epilogue warps
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int row_in_tile = q * 32 + lane;
    uint32_t it = 0;
    uint32_t flags = 0;
    for (int64_t t = blockIdx.x; t < L.total_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = decode_tile(L, t);
      const GemmProblem& P = L.prob[tc.p];
      const uint32_t buf = it & 1u;
      const uint32_t aph = (it >> 1) & 1u;
      if (!mbar_wait(&acc_full[buf], aph, L.status)) break;
      tc_fence_after();
      const int i = tc.tm * kBM + row_in_tile;
      float sumsq = 0.0f;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + c * 32, v);
        epilogue_chunk(P, tc, i, tc.tn * kBN + c * 32, v, flags, sumsq);
      }
      if (P.epi == EPI_SYRK) {
        // one partial per (tile, epilogue warp) in a fixed slot: the sum over
        // slots is taken later in a fixed order, so ||S||_F is reproducible
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
        if (lane == 0) P.part[static_cast<int64_t>(tc.mat) * P.part_ld + tc.lt * 4 + q] = sumsq;
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
    if (flags) atomicOr(L.status, flags);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(okls_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (L.total_tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(L.total_tiles < num_sms ? L.total_tiles : num_sms);
  okls_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace okls

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
//   warps 2-9        epilogue: tcgen05.ld of their 32 TMEM lanes and 128
//                    of the 256 columns, the fused OKLS arithmetic, global
//                    stores.
// The two accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.  All waits are bounded (okls_ptx.cuh) by the launch's limit;
// when one expires the kernel raises kStTimeout, every thread leaves its
// loop, the producer waits for its own copies still landing and the MMA
// thread for its own MMAs (neither of those two waits stops early because
// of another thread's timeout), and TMEM is freed before the CTA exits.
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
#include "okls_epilogue.cuh"
#include "okls_ptx.cuh"

namespace okls {

// The kernel body, shared by the two schedules:
//   kChain = false  one launch of up to kMaxProblems independent problems
//                   (okls_gemm_kernel; the problems in the parameter block);
//   kChain = true   a chain of dependent stages in one persistent launch
//                   (okls_chain_kernel; the problems in a device table): the
//                   producer waits, before loading a tile of stage s > 0,
//                   until its matrix's slot of stage s - 1 has dep_need
//                   completions, and each epilogue warp publishes its
//                   stores and adds one completion to its slot of stage s.
//                   Any status bit stops the chain: later stages must not
//                   run after a failure, as later launches skip it.
// Tiles go to CTAs with a static stride and each CTA visits them in
// increasing order; a tile only depends on tiles of earlier stages, which
// have lower indices, so the lowest unfinished tile can always proceed once
// every CTA is resident (the chain is launched cooperatively).
template <bool kChain>
__device__ __forceinline__ void gemm_body(const GemmProblem* probs, int nprob, int64_t total_tiles,
                                          const CUtensorMap* maps, uint32_t* status, int64_t wait_cycles,
                                          int64_t unloaded_tile, uint32_t* done, int nslot) {
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
  const long long lim = wait_cycles > 0 ? static_cast<long long>(wait_cycles) : kTimeoutCycles;
  const uint32_t abort_mask = kChain ? 0xFFFFFFFFu : kStTimeout;

  // An earlier stage of the step failed: leave W, S and P untouched.
  if (threadIdx.x == 0) *skip = (*reinterpret_cast<volatile uint32_t*>(status) != 0u);
  __syncthreads();
  if (*skip) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 256);
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
      if (!kChain)
        for (int p = 0; p < nprob; ++p)
          for (int s = 0; s < probs[p].nseg; ++s) {
            prefetch_tmap(maps + probs[p].amap[s]);
            prefetch_tmap(maps + probs[p].bmap[s]);
          }
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      int pi = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        // test hook: this tile's operands are never loaded, so its consumers'
        // waits run out with nothing of this CTA in flight
        if (t == unloaded_tile) break;
        const TileCoord tc = decode_tile(probs, nprob, t, pi);
        const GemmProblem& P = probs[tc.p];
        if (kChain) {
          if (*reinterpret_cast<volatile uint32_t*>(status) != 0u) break;
          if (P.dep_need > 0) {
            const uint32_t* ctr = done + static_cast<int64_t>(P.stage - 1) * nslot + P.dep_slot + tc.mat;
            if (!counter_wait(ctr, static_cast<uint32_t>(P.dep_need), status, lim)) break;
            // the operands were written by other CTAs' epilogues
            fence_proxy_async_global();
          }
        }
        const int nkb = (P.K + kBK - 1) / kBK;
        for (int sg = 0; sg < P.nseg && ok; ++sg) {
          const CUtensorMap* am = maps + P.amap[sg];
          const CUtensorMap* bm = maps + P.bmap[sg];
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, status, lim, abort_mask)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * kStageBytes;
            uint8_t* sb = sa + kStageABytes;
            mbar_expect_tx(&full[stage], kStageBytes);
            tma_load_3d(sa, am, &full[stage], kb * kBK, tc.tm * kBM, tc.mat);
            if (P.bmn) {
              // B stored K x N: four 64 (N) x 64 (K) boxes, 8 KB apart
#pragma unroll
              for (int c = 0; c < kBN / 64; ++c)
                tma_load_3d(sb + c * 8192, bm, &full[stage], tc.tn * kBN + c * 64, kb * kBK, tc.mat);
            } else {
              tma_load_3d(sb, bm, &full[stage], kb * kBK, tc.tn * kBN, tc.mat);
            }
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // make sure no bulk copy is still landing in shared memory at exit
      // (waits on this thread's own copies: the default limit, whatever the
      // status word says)
      const int64_t back = issued < kStages ? issued : kStages;
      for (int64_t q = 1; q <= back; ++q) {
        const int64_t idx = issued - q;
        const uint32_t s = static_cast<uint32_t>(idx % kStages);
        const uint32_t ph = static_cast<uint32_t>((idx / kStages) & 1);
        if (!mbar_wait_own(&full[s], ph, status)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      // a tile with at most 128 valid columns (the edge of a 5504-wide product)
      // runs N = 128 MMAs; the epilogue never reads the unused columns
      constexpr uint32_t idesc_k = idesc_f16_f32(kBM, kBN, false);
      constexpr uint32_t idesc_mn = idesc_f16_f32(kBM, kBN, true);
      constexpr uint32_t idesc_k_half = idesc_f16_f32(kBM, kBN / 2, false);
      constexpr uint32_t idesc_mn_half = idesc_f16_f32(kBM, kBN / 2, true);
      // descriptors of stage 0; stage s adds s * kStageBytes to the 16-byte
      // address field (shared memory stays below 2^18 bytes, so it never carries)
      const uint32_t s0 = smem_u32(smem);
      const uint64_t adesc0 = sw128_desc(s0);
      const uint64_t bdesc0_k = sw128_desc(s0 + kStageABytes);
      const uint64_t bdesc0_mn = sw128_mn_desc(s0 + kStageABytes);
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      uint32_t stage = 0, phase = 0, it = 0;
      int pi = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
        const TileCoord tc = decode_tile(probs, nprob, t, pi);
        const GemmProblem& P = probs[tc.p];
        const int nkb = ((P.K + kBK - 1) / kBK) * P.nseg;
        const uint32_t buf = it & 1u;
        const uint32_t aph = (it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, status, lim, abort_mask)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        const bool half_n = P.cols - tc.tn * kBN <= kBN / 2;
        const uint32_t id = P.bmn ? (half_n ? idesc_mn_half : idesc_mn) : (half_n ? idesc_k_half : idesc_k);
        const uint64_t bdesc0 = P.bmn ? bdesc0_mn : bdesc0_k;
        // K16 step of B: 16 rows of 128 B (MN-major) or 32 B (K-major)
        const uint64_t bstep = P.bmn ? (kUmmaK * 128) >> 4 : (kUmmaK * 2) >> 4;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, status, lim, abort_mask)) {
            ok = false;
            break;
          }
          tc_fence_after();
          umma_f16_kblock(d, adesc0 + stage * kStageDesc, bdesc0 + stage * kStageDesc, bstep, id, kb != 0 ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      // all MMAs retired before TMEM is released (this thread's own MMAs:
      // the default limit, whatever the status word says)
      umma_commit(drain);
      mbar_wait_own(drain, 0, status);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- epilogue warps
    // two warps per TMEM lane quarter (a warp reaches only the lanes of
    // quarter warp % 4), each taking 128 of the tile's 256 columns: short
    // tiles (K = 512) are bound by the epilogue, which this halves
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int half = (warp - 2) >> 2;        // which 128 of the tile's 256 columns
    const int row_in_tile = q * 32 + lane;
    uint32_t it = 0;
    uint32_t flags = 0;
    int pi = 0;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = decode_tile(probs, nprob, t, pi);
      const GemmProblem& P = probs[tc.p];
      const uint32_t buf = it & 1u;
      const uint32_t aph = (it >> 1) & 1u;
      if (!mbar_wait(&acc_full[buf], aph, status, lim, abort_mask)) break;
      tc_fence_after();
      const int i = tc.tm * kBM + row_in_tile;
      float sumsq = 0.0f;
#pragma unroll 1
      for (int c = half * 4; c < half * 4 + 4; ++c) {
        float v[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + c * 32, v);
        epilogue_chunk(P, tc, i, tc.tn * kBN + c * 32, v, flags, sumsq);
      }
      if (P.epi == EPI_SYRK) {
        // one partial per (tile, epilogue warp) in a fixed slot: the sum over
        // slots is taken later in a fixed order, so ||S||_F is reproducible
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
        if (lane == 0) P.part[static_cast<int64_t>(tc.mat) * P.part_ld + tc.lt * 8 + half * 4 + q] = sumsq;
      }
      if (P.epi == EPI_NS_LAST && tc.tm == 0 && tc.tn == 0 && q == 0 && half == 0 && lane == 0) {
        // the new root's scale, computed as the commit after the chain does
        const double cp = static_cast<double>(P.scal[static_cast<int64_t>(P.cp_slot) * P.scal_ld + tc.mat]);
        P.scal[static_cast<int64_t>(P.pi_slot) * P.scal_ld + tc.mat] = static_cast<float>(ldexp(1.0 / sqrt(cp), P.pi_exp));
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      if (kChain) {
        // publish this warp's stores to the other CTAs' TMA loads, then
        // count the warp's eighth of the tile as done
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0)
          red_release_gpu_add(done + static_cast<int64_t>(P.stage) * nslot + P.dep_slot + tc.mat, 1u);
      }
    }
    if (flags) atomicOr(status, flags);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

__global__ void __launch_bounds__(kGemmThreads, 1) okls_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  gemm_body<false>(L.prob, L.nprob, L.total_tiles, L.maps, L.status, L.wait_cycles, L.unloaded_tile, nullptr, 0);
}

__global__ void __launch_bounds__(kGemmThreads, 1) okls_chain_kernel(const __grid_constant__ ChainLaunch C) {
  gemm_body<true>(C.prob, C.nprob, C.total_tiles, C.maps, C.status, C.wait_cycles, C.unloaded_tile, C.done,
                  C.nslot);
}

cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t stream) {
  static PerDevice pd;
  const cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(okls_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  });
  if (e != cudaSuccess) return e;
  if (L.total_tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(L.total_tiles < num_sms ? L.total_tiles : num_sms);
  okls_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(L);
  return cudaGetLastError();
}

// The chain's CTAs wait on one another's tiles, so all of them must be
// resident at once: a cooperative launch of at most one CTA per SM (the
// kernel's shared memory admits no second one) guarantees it or fails.
cudaError_t launch_chain(const ChainLaunch& C, int num_sms, cudaStream_t stream) {
  static PerDevice pd;
  const cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(okls_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  });
  if (e != cudaSuccess) return e;
  if (C.total_tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(C.total_tiles < num_sms ? C.total_tiles : num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, okls_chain_kernel, C);
}

}  // namespace okls

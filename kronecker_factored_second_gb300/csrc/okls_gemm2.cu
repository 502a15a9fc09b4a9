// CTA-pair tcgen05 GEMM (sm_103a): the same problems and fused epilogues as
// okls_gemm.cu, on 256 x 256 output tiles computed by a cluster of two CTAs.
//
// CTA rank r of the pair owns output rows [tm*256 + r*128, +128) and keeps
// in its shared memory the matching 128 rows of A and 128 of the 256 rows of
// B (K-major), 32 KB per 64-deep K step, in a 7-stage ring.  The even CTA
// (leader) issues tcgen05.mma.cta_group::2 (M256 N256 K16), which reads A and
// B from both CTAs and writes each CTA's 128 accumulator rows into its own
// Tensor Memory.  Compared with one CTA per 128 x 256 tile this halves the B
// bytes every SM loads and stores (64 instead of 94 B per MMA cycle at full
// rate) and deepens the ring from 4 x 48 KB to 7 x 32 KB.
//
// Barriers (per CTA, same offsets in both):
//   full[s]      leader only; counts both CTAs' TMA bytes of stage s (each
//                CTA's loads name the leader's barrier, .cta_group::2)
//   empty[s]     both; the leader's commit arrives on both (multicast)
//   acc_full[b]  both; accumulator b is ready (multicast commit)
//   acc_empty[b] leader only; 8 epilogue warps (4 per CTA) arrive
// All waits are bounded (okls_ptx.cuh); the pair decides together whether
// an earlier failure means the launch must do nothing.
#include "okls_epilogue.cuh"
#include "okls_ptx.cuh"

namespace okls {

constexpr int kPairStages = 7;
constexpr int kPairStageA = 128 * kBK * 2;  // 16 KB
constexpr int kPairStageB = 128 * kBK * 2;  // 16 KB
constexpr int kPairStageBytes = kPairStageA + kPairStageB;
constexpr int kPairSmem = kPairStages * kPairStageBytes + 1024 + 256;
static_assert(kPairSmem <= 232448, "pair ring exceeds shared memory");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    okls_gemm_pair_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStageBytes);
  uint64_t* empty = full + kPairStages;
  uint64_t* acc_full = empty + kPairStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* skip = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int64_t pair_id = blockIdx.x >> 1;
  const int64_t npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    *skip = (*reinterpret_cast<volatile uint32_t*>(L.status) != 0u) ? 1u : 0u;
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  cluster_sync();
  // both CTAs follow the leader's decision, so neither waits for the other
  const uint32_t skip_pair = ld_shared_cluster_u32(mapa_shared(smem_u32(skip), 0));
  cluster_sync();
  if (skip_pair) return;

  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer (both CTAs)
      for (int p = 0; p < L.nprob; ++p)
        for (int s = 0; s < L.prob[p].nseg; ++s) {
          prefetch_tmap(L.maps + L.prob[p].amap[s]);
          prefetch_tmap(L.maps + L.prob[p].bmap_pair[s]);
        }
      const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = pair_id; t < L.total_tiles && ok; t += npairs) {
        const TileCoord tc = decode_tile<256>(L, t);
        const GemmProblem& P = L.prob[tc.p];
        const int nkb = (P.K + kBK - 1) / kBK;
        const int row_a = tc.tm * 256 + static_cast<int>(rank) * 128;
        const int row_b = tc.tn * kBN + static_cast<int>(rank) * 128;
        for (int sg = 0; sg < P.nseg && ok; ++sg) {
          const CUtensorMap* am = L.maps + P.amap[sg];
          const CUtensorMap* bm = L.maps + P.bmap_pair[sg];  // 128-row boxes: half of B
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, L.status)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * kPairStageBytes;
            uint8_t* sb = sa + kPairStageA;
            if (leader) mbar_expect_tx(&full[stage], 2 * kPairStageBytes);
            const uint32_t fb = full_leader + stage * 8u;
            tma_load_3d_pair(sa, am, fb, kb * kBK, row_a, tc.mat);
            if (P.bmn) {
              // this CTA's 128 columns of a K x N B: two 64 x 64 boxes, 8 KB apart
              tma_load_3d_pair(sb, bm, fb, row_b, kb * kBK, tc.mat);
              tma_load_3d_pair(sb + 8192, bm, fb, row_b + 64, kb * kBK, tc.mat);
            } else {
              tma_load_3d_pair(sb, bm, fb, kb * kBK, row_b, tc.mat);
            }
            ++issued;
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // the leader's full barriers count both CTAs' bytes: once the last
      // stages completed, no copy is still landing in either CTA
      if (leader) {
        const int64_t back = issued < kPairStages ? issued : kPairStages;
        for (int64_t q = 1; q <= back; ++q) {
          const int64_t idx = issued - q;
          const uint32_t s = static_cast<uint32_t>(idx % kPairStages);
          const uint32_t ph = static_cast<uint32_t>((idx / kPairStages) & 1);
          if (!mbar_wait_cluster(&full[s], ph, L.status)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idesc_k = idesc_f16_f32(256, kBN, false);
      constexpr uint32_t idesc_mn = idesc_f16_f32(256, kBN, true);
      const uint32_t s0 = smem_u32(smem);
      const uint64_t adesc0 = sw128_desc(s0);
      const uint64_t bdesc0_k = sw128_desc(s0 + kPairStageA);
      const uint64_t bdesc0_mn = sw128_mn_desc(s0 + kPairStageA);
      constexpr uint64_t kStageDesc = kPairStageBytes >> 4;
      uint32_t stage = 0, phase = 0, it = 0;
      bool ok = true;
      for (int64_t t = pair_id; t < L.total_tiles && ok; t += npairs, ++it) {
        const TileCoord tc = decode_tile<256>(L, t);
        const GemmProblem& P = L.prob[tc.p];
        const int nkb = ((P.K + kBK - 1) / kBK) * P.nseg;
        const uint32_t buf = it & 1u;
        const uint32_t aph = (it >> 1) & 1u;
        if (!mbar_wait_cluster(&acc_empty[buf], aph ^ 1u, L.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, L.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          umma_f16_pair_kblock(d, adesc0 + stage * kStageDesc, (P.bmn ? bdesc0_mn : bdesc0_k) + stage * kStageDesc,
                               P.bmn ? (kUmmaK * 128) >> 4 : (kUmmaK * 2) >> 4, P.bmn ? idesc_mn : idesc_k,
                               kb != 0 ? 1u : 0u);
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&acc_full[buf], 0x3);
      }
      umma_commit_pair(drain, 0x1);
      mbar_wait(drain, 0, L.status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- epilogue warps (both CTAs)
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
    uint32_t it = 0;
    uint32_t flags = 0;
    for (int64_t t = pair_id; t < L.total_tiles; t += npairs, ++it) {
      const TileCoord tc = decode_tile<256>(L, t);
      const GemmProblem& P = L.prob[tc.p];
      const uint32_t buf = it & 1u;
      const uint32_t aph = (it >> 1) & 1u;
      if (!mbar_wait(&acc_full[buf], aph, L.status)) break;
      tc_fence_after();
      const int i = tc.tm * 256 + static_cast<int>(rank) * 128 + row_in_tile;
      float sumsq = 0.0f;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + c * 32, v);
        epilogue_chunk(P, tc, i, tc.tn * kBN + c * 32, v, flags, sumsq);
      }
      if (P.epi == EPI_SYRK) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
        if (lane == 0)
          P.part[static_cast<int64_t>(tc.mat) * P.part_ld + tc.lt * 8 + static_cast<int64_t>(rank) * 4 + q] = sumsq;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty_leader + buf * 8u);
    }
    if (flags) atomicOr(L.status, flags);
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

cudaError_t launch_gemm_pair(const GemmLaunch& L, int num_sms, cudaStream_t stream) {
  static PerDevice pd;
  const cudaError_t e = once_per_device(pd, [](int) {
    return cudaFuncSetAttribute(okls_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  });
  if (e != cudaSuccess) return e;
  if (L.total_tiles <= 0) return cudaSuccess;
  const int64_t pairs = L.total_tiles < num_sms / 2 ? L.total_tiles : num_sms / 2;
  okls_gemm_pair_kernel<<<static_cast<int>(2 * pairs), kGemmThreads, kPairSmem, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace okls

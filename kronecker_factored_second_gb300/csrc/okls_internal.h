// Internal structures shared by the host planner and the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace okls {

// Host-side set-up that must run once per device for one call site (the
// kernels' shared-memory opt-ins, occupancy queries): `set(device)` runs for
// the caller's current device unless it already succeeded there.  Safe to
// call from several host threads; devices past 63 are set up on every call.
struct PerDevice {
  std::mutex mu;
  uint64_t done = 0;  // bit d: device d is set up
};
template <class F>
inline cudaError_t once_per_device(PerDevice& pd, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  std::lock_guard<std::mutex> lock(pd.mu);
  if (pd.done & bit) return cudaSuccess;
  e = set(dev);
  if (e == cudaSuccess) pd.done |= bit;
  return e;
}

// ----------------------------------------------------------------- tiling
constexpr int kBM = 128;        // output rows per tile (UMMA M, one TMEM lane each)
constexpr int kBN = 256;        // output cols per tile (UMMA N, TMEM columns)
constexpr int kBK = 64;         // K per pipeline stage: 64 fp16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;      // K of one tcgen05.mma kind::f16
constexpr int kStages = 4;      // smem ring depth
constexpr int kStageABytes = kBM * kBK * 2;   // 16 KB
constexpr int kStageBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kStageABytes + kStageBBytes;
constexpr int kGemmThreads = 320;             // warp0 TMA, warp1 MMA, warps2-9 epilogue
constexpr int kTmemCols = 512;                // two 256-column fp32 accumulators
constexpr int kGemmSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr int kMaxProblems = 6;
constexpr int kMaxSeg = 3;                    // K segments (split mode: hi*hi, hi*lo, lo*hi)
// Raster of non-symmetric products: output tiles go in groups of group_m
// row blocks, column by column inside a group, so a group's A row panels stay
// in L2 while its columns pass and each B column panel is read once per
// group.  group_m is chosen per problem on the host: the largest height
// (groups of equal size) whose A panels plus the B panels of one wave of
// tiles fit kRasterL2Bytes.
constexpr double kRasterL2Bytes = 64.0 * 1024 * 1024;

// Binary16 operand headroom (power of two) of the Newton-Schulz iterates.
constexpr int kHeadroom = 12;

// Per-matrix scalar slots (float), laid out [slot][batch].
enum ScalarSlot {
  SC_SUMSQ_G = 0,    // sum G^2 of this step            (zeroed every step)
  SC_SUMSQ_N = 1,    // sum N^2                          (zeroed every step)
  SC_SUMSQ_SA = 2,   // ||S_a||_F^2                      (zeroed every step)
  SC_SUMSQ_SB = 3,   // ||S_b||_F^2                      (zeroed every step)
  SC_GSCALE = 4,     // Ghat = G * gscale (power of two)
  SC_NSCALE = 5,     // Nhat = N * nscale (power of two)
  SC_ALPHA_SA = 6,   // S_a += alpha_a * (Xhat_b Xhat_b^T)
  SC_ALPHA_SB = 7,   // S_b += alpha_b * (Xhat_a^T Xhat_a)
  SC_PI_A = 8,       // P_a = pi_a * Phat_a              (persistent)
  SC_PI_B = 9,       // P_b = pi_b * Phat_b              (persistent)
  SC_CPRIME_A = 10,  // normaliser c' of S_a
  SC_CPRIME_B = 11,
  SC_PSCALE_A = 12,  // fp32 P_a = acc * pscale_a at the last product
  SC_PSCALE_B = 13,
  SC_RSCALE_A = 14,  // root S_a^1/2 = acc * rscale_a (debug root output)
  SC_RSCALE_B = 15,
  SC_UCOEF = 16,     // U = acc_U * ucoef
  SC_COUNT = 17
};

// Status word bits (mirror of okls.h).
constexpr uint32_t kStNonfiniteInput = 0x1u;
constexpr uint32_t kStNonfiniteIter = 0x2u;
constexpr uint32_t kStNonfiniteUpdate = 0x4u;
constexpr uint32_t kStTimeout = 0x8u;

// ----------------------------------------------------------------- epilogues
enum EpiKind : int32_t {
  EPI_X16 = 0,       // out16 = acc * alpha (row-major)          [X_b, X_a^T, Q]
  EPI_SYRK = 1,      // S = beta2 S + alpha_b acc + eps I, symmetric tiles, sum S^2
  EPI_NS_T = 2,      // T = a' I + b' acc  -> fp16 row + transposed (+lo)
  EPI_NS_SCALE = 3,  // out = acc * alpha  -> fp16 row + transposed (+lo)
  EPI_NS_LAST = 4,   // P32 = acc * pscale_b ; Phat = acc * alpha (row + transposed)
  EPI_UPDATE = 5,    // W = W * decay - coef_b * acc
  EPI_ROOT = 6       // root32 = acc * rscale_b (debug)
};

struct GemmProblem {
  // operands: K segments, each a pair of tensor-map indices (A: box 128 rows,
  // B: box 256 rows) into the handle's descriptor table
  int32_t nseg;
  int32_t amap[kMaxSeg];        // A descriptors, 128-row boxes
  int32_t bmap[kMaxSeg];        // B descriptors: K-major 256-row boxes, or MN-major 64x64 boxes
                                // when bmn
  int32_t bmn;                  // 1: B is stored K x N row-major (MN-major operand)
  int32_t rows, cols, K;        // output rows (A rows), cols (B rows), K
  int32_t batch;
  int32_t tiles_m, tiles_n;
  int32_t sym;                  // 1: only tiles touching the upper triangle
  int32_t epi;
  int64_t tiles_per_mat;
  int64_t tile_begin;           // first linear tile of this problem in the launch
  // exact division of tile indices (< 2^31) by tiles_per_mat, by the raster
  // group span group_m * tiles_n, by group_m and by the height of the last
  // (shorter) group: q = (n * mul) >> shift (host-computed)
  uint32_t tpm_mul, tpm_shift, span_mul, span_shift;
  int32_t group_m, last_gm;
  uint32_t gm_mul, gm_shift, lgm_mul, lgm_shift;
  // epilogue
  void* out_hi;                 // fp16 row-major
  void* out_hi_t;               // fp16 transposed (may be null)
  void* out_lo;                 // fp16 row-major low half (split outputs)
  void* out_lo_t;
  int64_t ld16;                 // row pitch (elements) of fp16 outputs
  int64_t mat16;                // elements per matrix of fp16 outputs
  float* out32;                 // fp32 output / state (S, P, W fp32)
  void* w;                      // parameter (EPI_UPDATE), fp32 or bf16
  int32_t w_bf16;
  int64_t ld32, mat32;          // fp32 / W row pitch and matrix stride (elements)
  float* scal;                  // per-matrix scalar table base [SC_COUNT][scal_ld]
  int32_t scal_ld;              // matrices per slot row of the table
  int32_t scal_slot;            // slot read by this epilogue (alpha_b, pscale, coef)
  float* part;                  // EPI_SYRK: per-(tile, warp) partial sums of S^2
  int64_t part_ld;              // partial slots per matrix (>= 4 * tiles_per_mat)
  float alpha, beta, gamma, delta;  // kind-specific constants
  int32_t split_out;            // 1: also write lo halves
  int32_t check_finite;         // 1: raise kStNonfiniteIter on non-finite acc
  // EPI_NS_LAST: the root's scale pi = 2^pi_exp / sqrt(c') is written with
  // the root (slot pi_slot, c' from slot cp_slot) by the tile at (0, 0), so
  // a matrix's binary16 root and its scale always change together
  int32_t pi_slot, cp_slot, pi_exp;
  // chain launches (okls_chain_kernel) only: the problem's stage, the
  // completion-counter slot of its matrix 0 (a factor's matrix b uses
  // dep_slot + b), and how many completions (8 per tile, one per epilogue
  // warp) that slot must reach in the previous stage before a tile of this
  // problem may load its operands (0: no dependency)
  int32_t stage;
  int32_t dep_slot;
  int32_t dep_need;
};

// Division by an invariant d >= 1 for dividends n < 2^31: with
// s = ceil(log2 d) and mul = ceil(2^(31+s) / d) < 2^32, floor(n * mul / 2^(31+s))
// = floor(n / d), because the rounding of mul adds less than n / 2^(31+s) < 2^-s
// <= 1/d to n/d (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994).
__host__ __device__ inline void fastdiv_make(uint32_t d, uint32_t* mul, uint32_t* shift) {
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  const unsigned long long num = 1ull << (31 + s);
  *mul = static_cast<uint32_t>((num + d - 1) / d);
  *shift = 31 + s;
}

__host__ __device__ __forceinline__ uint32_t fastdiv(uint32_t n, uint32_t mul, uint32_t shift) {
  return static_cast<uint32_t>((static_cast<unsigned long long>(n) * mul) >> shift);
}

// A chain of dependent GEMM stages in one persistent launch: the stages'
// problems live in a device table (stage-major, tile_begin counting through
// all stages); a tile of stage s > 0 waits until its matrix's slot of stage
// s - 1 has reached dep_need completions, and every epilogue warp adds one
// completion to its slot of stage s when its stores are done.
constexpr int kChainMaxProblems = 256;
struct ChainLaunch {
  const GemmProblem* prob;      // device table
  int32_t nprob;
  int32_t nslot;                // counter slots per stage
  int64_t total_tiles;
  uint32_t* done;               // [stages][nslot] completion counters, zero when the launch starts
  const CUtensorMap* maps;
  uint32_t* status;
  int64_t wait_cycles;          // as GemmLaunch
  int64_t unloaded_tile;
};

struct GemmLaunch {
  GemmProblem prob[kMaxProblems];
  int32_t nprob;
  int64_t total_tiles;
  const CUtensorMap* maps;      // device table of descriptors (64-byte aligned)
  uint32_t* status;
  int64_t wait_cycles;          // limit of every pipeline wait (<= 0: the default, ~2 s of SM clock)
  int64_t unloaded_tile;        // test hook: the producer stops before this linear tile (-1: none)
};

}  // namespace okls

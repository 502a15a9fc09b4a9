// C ABI of the OKLS step: validation, workspace planning, TMA descriptors and
// the launch sequence of one step (see include/okls.h for the contract).
//
// Step (page "Online KL Shampoo", "How it works"), per same-shape batch:
//   1. momentum statistics          k_momentum_stats, k_coeffs_pre
//   2. M_t, Ghat, Ghat^T, Nhat^T    k_pack
//   3. X_b = G P_b, X_a^T = G^T P_a^T             GEMM (EPI_X16)
//      (B operands stored K x N are read MN-major, so every binary16 matrix
//      is kept in one row-major layout; only Ghat^T is materialised)
//   4. S_a, S_b EMAs (+ ||S||_F^2)                 GEMM (EPI_SYRK, upper triangle;
//      the normaliser of step 5 writes the mirrored lower triangle)
//   5. normalisers, Y_0, T_0, Z_1                  k_coeffs_post, k_normalise
//   6. coupled Newton-Schulz, both factors         19 GEMM launches, 27 products
//   7. Q = P_a N                                    GEMM (EPI_X16)
//   8. U = Q P_b and the parameter update          GEMM (EPI_UPDATE)
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/okls.h"
#include "okls_internal.h"
#include "okls_kernels.h"

using namespace okls;

namespace {

thread_local std::string g_err;

okls_status fail(okls_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

#define OKLS_CK(call)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(OKLS_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                                  \
  } while (0)

// ------------------------------------------------------------------ schedule
// Minimax odd cubic q(s) = a s + b s^3 of 1 on [l, u] (equioscillation at l,
// sqrt(D/3), u with D = u^2 + u l + l^2), next interval [q(l), q(sqrt(D/3))];
// exponents z_k = ceil(log2(prod_{j<k} a_j)).
struct Sched {
  int iters = 0;
  std::vector<double> a, b;
  std::vector<int> z;
};

Sched make_schedule(int iters, double lo) {
  Sched s;
  s.iters = iters;
  double l = lo, u = 1.0, prod = 1.0;
  s.z.push_back(0);
  for (int k = 0; k < iters; ++k) {
    const double D = u * u + u * l + l * l;
    const double a = 2.0 / (l * u * (u + l) / D + (2.0 / 3.0) * std::sqrt(D / 3.0));
    const double b = -a / D;
    s.a.push_back(a);
    s.b.push_back(b);
    prod *= a;
    s.z.push_back(static_cast<int>(std::ceil(std::log2(prod))));
    const double ss = std::sqrt(D / 3.0);
    const double nl = a * l + b * l * l * l, nu = a * ss + b * ss * ss * ss;
    l = nl;
    u = nu;
  }
  return s;
}

// variance of the Nesterov combination for iid unit-variance gradients:
// v_t = (1-b)^2 [ (1+b)^2 + sum_{k=2}^{t} b^{2k} ]; kappa = v_t^-1/2
double variance_kappa(double b, int64_t t) {
  const double b2 = b * b;
  double tail = 0.0;
  if (t >= 2) tail = (b2 < 1.0) ? b2 * b2 * (1.0 - std::pow(b2, static_cast<double>(t - 1))) / (1.0 - b2) : 0.0;
  const double v = (1.0 - b) * (1.0 - b) * ((1.0 + b) * (1.0 + b) + tail);
  return 1.0 / std::sqrt(v);
}

// ------------------------------------------------------------ TMA encoding
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

constexpr int kMaxMaps = 128;
constexpr int kMNBox = 64;  // descriptor code of a 64 x 64 MN-major box
constexpr size_t kMapTableBytes = kMaxMaps * sizeof(CUtensorMap);

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// tiles (128 x 256) of a symmetric (upper-triangle) d x d product: row
// block tm holds column blocks floor(tm / 2) .. tiles_n-1
int64_t sym_tiles(int64_t d) {
  const int64_t tm_n = (d + kBM - 1) / kBM, tn_n = (d + kBN - 1) / kBN;
  constexpr int div = kBN / kBM;
  int64_t c = 0;
  for (int64_t tm = 0; tm < tm_n; ++tm) c += tn_n - tm / div;
  return c;
}

// partial sums of S^2 one symmetric product writes: 8 epilogue warps per tile
int64_t syrk_parts(int64_t d) { return 8 * sym_tiles(d); }

// fixed partial slots per matrix for ||S||_F^2 (the product's tiles, or the
// blocks of the standalone reduction)
int64_t factor_parts(int64_t d) { return std::max(syrk_parts(d), static_cast<int64_t>(sumsq_parts(d * d))); }

// A batch of binary16 matrices (rows x cols, row pitch ld) with two TMA
// descriptors: box 128 rows (A operand) and box 256 rows (B operand).
struct Buf {
  __half* p = nullptr;
  int64_t rows = 0, cols = 0, ld = 0, batch = 0;
  int mapA = -1, mapB = -1;  // K-major boxes: 128 and 256 rows of 64 columns
  int mapMN = -1;            // MN-major box: 64 columns x 64 rows
  int64_t mat() const { return rows * ld; }
};

struct Planner {
  uint8_t* base = nullptr;  // null: sizing pass
  size_t off = 0;
  std::vector<CUtensorMap> maps;
  std::vector<int> boxes;  // rows of each descriptor's box (128 or 256)
  okls_status err = OKLS_OK;

  void* take(size_t bytes, size_t align = 256) {
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), static_cast<int64_t>(align)));
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }

  // box_rows 128 / 256: K-major operand tiles (64 columns); box_rows kMNBox:
  // MN-major 64 x 64 tiles.  The recorded code is what the launch check reads.
  int make_map(void* ptr, int64_t rows, int64_t cols, int64_t ld, int64_t batch, int box_rows) {
    if (!base) return 0;
    if (static_cast<int>(maps.size()) >= kMaxMaps) {
      err = fail(OKLS_ERR_UNSUPPORTED, "descriptor table full");
      return -1;
    }
    auto fn = encode_fn();
    if (!fn) {
      err = fail(OKLS_ERR_NO_DEVICE, "cuTensorMapEncodeTiled unavailable");
      return -1;
    }
    CUtensorMap m;
    memset(&m, 0, sizeof(m));
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(rows * ld * 2)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows == kMNBox ? 64 : box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, ptr, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      err = fail(OKLS_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld ld=%lld",
                 static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols),
                 static_cast<long long>(ld));
      return -1;
    }
    maps.push_back(m);
    boxes.push_back(box_rows);
    return static_cast<int>(maps.size()) - 1;
  }

  Buf buf16(int64_t rows, int64_t cols, int64_t batch) {
    Buf b;
    b.rows = rows;
    b.cols = cols;
    b.ld = round_up(cols, 8);
    b.batch = batch;
    b.p = static_cast<__half*>(take(static_cast<size_t>(b.mat() * batch * 2)));
    b.mapA = make_map(b.p, rows, cols, b.ld, batch, kBM);
    b.mapB = make_map(b.p, rows, cols, b.ld, batch, kBN);
    b.mapMN = make_map(b.p, rows, cols, b.ld, batch, kMNBox);
    return b;
  }
};

// One Newton-Schulz factor (a batch of d x d matrices).
struct Factor {
  int d = 0;
  int batch = 0;
  float* S = nullptr;       // fp32 input
  bool S_upper_only = false;  // S comes from the factor product: upper triangle only
  float* P32 = nullptr;     // fp32 output
  float* root32 = nullptr;  // debug root output
  Buf Ph[2];                         // binary16 P (hi, lo), row-major
  Buf Y[2][2], Z[2][2], T[2];        // iterates [ping-pong][hi, lo], row-major
  bool split = false;
  int slot_sumsq = 0, slot_cprime = 0, slot_pi = 0, slot_pscale = 0, slot_rscale = 0;
};

void plan_factor(Planner& pl, Factor& f, int d, int batch, bool split) {
  f.d = d;
  f.batch = batch;
  f.split = split;
  const int nl = split ? 2 : 1;
  for (int l = 0; l < nl; ++l) f.Ph[l] = pl.buf16(d, d, batch);
  for (int pp = 0; pp < 2; ++pp)
    for (int l = 0; l < nl; ++l) {
      f.Y[pp][l] = pl.buf16(d, d, batch);
      f.Z[pp][l] = pl.buf16(d, d, batch);
    }
  for (int l = 0; l < nl; ++l) f.T[l] = pl.buf16(d, d, batch);
}

int g_num_sms[64] = {0};

okls_status device_sms(int* out) {
  int dev = 0;
  OKLS_CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(OKLS_ERR_NO_DEVICE, "device index %d", dev);
  if (g_num_sms[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    OKLS_CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    OKLS_CK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    OKLS_CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (major != 10 || minor != 3)
      return fail(OKLS_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                  minor);
    g_num_sms[dev] = sms;
  }
  *out = g_num_sms[dev];
  return OKLS_OK;
}

// ------------------------------------------------------------ profiling
// Counts every kernel a step launches; with timing on, brackets each GEMM
// launch with CUDA events on the launching stream and records its
// algorithmic FLOPs (dense: 2 M N K per segment; symmetric: M (M+1) K, the
// upper triangle only).
struct Prof {
  bool timing = false;
  struct Rec {
    cudaEvent_t a, b;
    double flops;
    bool ns;
    bool bw;  // a bandwidth kernel (time goes to bw_ms)
  };
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  std::vector<Rec> recs;
  int64_t kernels = 0, gemm_launches = 0, ns_launches = 0, bw_launches = 0;
  double gemm_flops = 0.0, ns_flops = 0.0, bw_bytes = 0.0;

  cudaEvent_t next_event() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
  ~Prof() {
    for (cudaEvent_t e : pool) cudaEventDestroy(e);
  }
};

thread_local Prof* g_prof = nullptr;  // set for the duration of okls_step
thread_local const std::vector<int>* g_boxes = nullptr;  // box rows of each descriptor
thread_local bool g_in_ns = false;

void note_kernels(int n) {
  if (g_prof) g_prof->kernels += n;
}

// Launch one bandwidth kernel through `launch` (returns cudaError_t), counting
// it and its algorithmic DRAM bytes, bracketed by events when timing is on.
template <class F>
okls_status bw_launch(double bytes, cudaStream_t st, F&& launch) {
  Prof* pf = g_prof;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (pf && pf->timing) {
    ea = pf->next_event();
    eb = pf->next_event();
    if (ea) OKLS_CK(cudaEventRecord(ea, st));
  }
  OKLS_CK(launch());
  if (pf) {
    if (ea && eb) {
      OKLS_CK(cudaEventRecord(eb, st));
      pf->recs.push_back({ea, eb, 0.0, false, true});
    }
    pf->kernels += 1;
    pf->bw_launches += 1;
    pf->bw_bytes += bytes;
  }
  return OKLS_OK;
}

struct ProfScope {
  explicit ProfScope(Prof* p) { g_prof = p; }
  ~ProfScope() { g_prof = nullptr; }
};

struct BoxScope {
  explicit BoxScope(const std::vector<int>* b) { g_boxes = b; }
  ~BoxScope() { g_boxes = nullptr; }
};

// Wait limit of the GEMM launches of the current call (0: the kernels'
// default) and the test hook that leaves one tile's operands unloaded
// (okls_set_wait_limit).
struct WaitSetting {
  int64_t cycles = 0;
  int64_t unloaded_tile = -1;
};
thread_local WaitSetting g_wait;

struct WaitScope {
  explicit WaitScope(const WaitSetting& w) { g_wait = w; }
  ~WaitScope() { g_wait = WaitSetting(); }
};

// ------------------------------------------------------------ GEMM launches
// Output buffers must cover the problem's rows x cols (and cols x rows for the
// transposed copy, which shares the pitch); a violation is a planning bug.
thread_local bool g_plan_error = false;

// Raster group height of a non-symmetric problem (see kRasterL2Bytes): the
// largest height, in groups of equal size, for which the group's A row
// panels and the B column panels one wave of `sms` tiles spans fit the L2
// budget.  OKLS_GROUP_M=<rows> overrides it (tuning experiments).
int env_group_m() {
  static const int v = [] {
    const char* e = getenv("OKLS_GROUP_M");
    return e ? atoi(e) : 0;
  }();
  return v;
}

void raster_plan(GemmProblem& p, int sms) {
  const int tm = p.tiles_m;
  int gm = 0;
  if (env_group_m() > 0) {
    gm = std::min(env_group_m(), tm);
  } else {
    const double a_panel = static_cast<double>(kBM) * p.K * 2.0 * p.nseg;  // one row block of A
    const double b_panel = static_cast<double>(kBN) * p.K * 2.0 * p.nseg;  // one column block of B
    for (int groups = 1; groups <= tm && gm == 0; ++groups) {
      const int h = (tm + groups - 1) / groups;
      const int wave_cols = (sms + h - 1) / h;
      if (h * a_panel + std::min(wave_cols, p.tiles_n) * b_panel <= kRasterL2Bytes) gm = h;
    }
    // nothing fits: the height whose wave footprint h a + (sms / h) b is
    // smallest, h = sqrt(sms b / a) = sqrt(2 sms)
    if (gm == 0) gm = std::min(tm, static_cast<int>(std::lround(std::sqrt(2.0 * sms))));
  }
  if (gm < 1) gm = 1;
  p.group_m = gm;
  p.last_gm = tm % gm == 0 ? gm : tm % gm;
  fastdiv_make(static_cast<uint32_t>(gm * p.tiles_n), &p.span_mul, &p.span_shift);
  fastdiv_make(static_cast<uint32_t>(gm), &p.gm_mul, &p.gm_shift);
  fastdiv_make(static_cast<uint32_t>(p.last_gm), &p.lgm_mul, &p.lgm_shift);
}

struct LaunchBuilder {
  GemmLaunch L;
  LaunchBuilder() { memset(&L, 0, sizeof(L)); }

  // D = sum over segments of A_seg * op(B_seg); split: (hi,hi), (hi,lo), (lo,hi).
  // op(B) = B^T for K-major B (stored N x K), B for MN-major B (stored K x N).
  GemmProblem& add(const Buf* A, const Buf* B, bool split, int rows, int cols, int K, int batch, int epi,
                   bool sym, bool bmn = false) {
    GemmProblem& p = L.prob[L.nprob++];
    memset(&p, 0, sizeof(p));
    p.bmn = bmn ? 1 : 0;
    auto bm = [&](const Buf& x) { return bmn ? x.mapMN : x.mapB; };
    p.nseg = split ? 3 : 1;
    p.amap[0] = A[0].mapA;
    p.bmap[0] = bm(B[0]);
    if (split) {
      p.amap[1] = A[0].mapA;
      p.bmap[1] = bm(B[1]);
      p.amap[2] = A[1].mapA;
      p.bmap[2] = bm(B[0]);
    }
    p.rows = rows;
    p.cols = cols;
    p.K = K;
    p.batch = batch;
    p.sym = sym ? 1 : 0;
    p.epi = epi;
    return p;
  }

  // D = A * op(B_hi + B_lo): two K segments when `split`, else one
  GemmProblem& add_bsplit(const Buf& A, const Buf* B, bool split, int rows, int cols, int K, int batch, int epi,
                          bool bmn = false) {
    GemmProblem& p = add(&A, B, false, rows, cols, K, batch, epi, false, bmn);
    if (split) {
      p.nseg = 2;
      p.amap[1] = A.mapA;
      p.bmap[1] = bmn ? B[1].mapMN : B[1].mapB;
    }
    return p;
  }

  // D = (A_hi + A_lo) * op(B)
  GemmProblem& add_asplit(const Buf* A, const Buf& B, bool split, int rows, int cols, int K, int batch, int epi,
                          bool bmn = false) {
    GemmProblem& p = add(A, &B, false, rows, cols, K, batch, epi, false, bmn);
    if (split) {
      p.nseg = 2;
      p.amap[1] = A[1].mapA;
      p.bmap[1] = p.bmap[0];
    }
    return p;
  }

  // Validate the problems, order them (longest K first) and lay out their
  // tiles from linear tile `base` on; *flops gets their algorithmic FLOPs.
  okls_status prepare(int sms, int64_t base, double* flops) {
    if (g_plan_error) {
      g_plan_error = false;
      return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: output buffer smaller than a GEMM problem");
    }
    for (int i = 0; i < L.nprob; ++i) {
      const GemmProblem& p = L.prob[i];
      if ((p.epi == EPI_SYRK || p.epi == EPI_NS_LAST || p.epi == EPI_ROOT) && (p.out32 == nullptr || p.ld32 < p.cols))
        return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: fp32 output");
      if (p.epi == EPI_UPDATE && (p.w == nullptr || p.ld32 < p.cols || p.mat32 < static_cast<int64_t>(p.rows) * p.ld32))
        return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: parameter output");
    }
    // longest K first so the expensive tiles start in the first wave
    std::stable_sort(L.prob, L.prob + L.nprob, [](const GemmProblem& x, const GemmProblem& y) {
      return static_cast<int64_t>(x.K) * x.nseg > static_cast<int64_t>(y.K) * y.nseg;
    });
    // every TMA box must match the ring slot it lands in
    if (g_boxes) {
      const int nb = static_cast<int>(g_boxes->size());
      auto box = [&](int idx) { return (idx >= 0 && idx < nb) ? (*g_boxes)[idx] : -1; };
      for (int i = 0; i < L.nprob; ++i)
        for (int sg = 0; sg < L.prob[i].nseg; ++sg)
          if (box(L.prob[i].amap[sg]) != kBM || box(L.prob[i].bmap[sg]) != (L.prob[i].bmn ? kMNBox : kBN))
            return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: descriptor box sizes");
    } else {
      return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: descriptor table not bound");
    }
    int64_t t = base;
    for (int i = 0; i < L.nprob; ++i) {
      GemmProblem& p = L.prob[i];
      p.tiles_m = (p.rows + kBM - 1) / kBM;
      p.tiles_n = (p.cols + kBN - 1) / kBN;
      p.tiles_per_mat = p.sym ? sym_tiles(p.rows) : static_cast<int64_t>(p.tiles_m) * p.tiles_n;
      if (p.epi == EPI_SYRK && (p.part == nullptr || p.part_ld < syrk_parts(p.rows)))
        return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: partial-sum slots");
      p.tile_begin = t;
      t += p.tiles_per_mat * p.batch;
      fastdiv_make(static_cast<uint32_t>(p.tiles_per_mat), &p.tpm_mul, &p.tpm_shift);
      raster_plan(p, sms);
    }
    // the kernels decode tile indices in 32 bits
    if (t >= (int64_t(1) << 31)) return fail(OKLS_ERR_UNSUPPORTED, "more than 2^31 output tiles in one launch");
    L.total_tiles = t;
    double f = 0.0;
    for (int i = 0; i < L.nprob; ++i) {
      const GemmProblem& p = L.prob[i];
      const double mn =
          p.sym ? static_cast<double>(p.rows) * (p.rows + 1) * 0.5 : static_cast<double>(p.rows) * p.cols;
      f += 2.0 * mn * p.K * p.batch * p.nseg;
    }
    *flops = f;
    return OKLS_OK;
  }

  okls_status go(const CUtensorMap* maps, uint32_t* status, int sms, cudaStream_t st) {
    double flops = 0.0;
    okls_status s0 = prepare(sms, 0, &flops);
    if (s0 != OKLS_OK) return s0;
    L.maps = maps;
    L.status = status;
    L.wait_cycles = g_wait.cycles;
    L.unloaded_tile = g_wait.unloaded_tile;
    Prof* pf = g_prof;
    cudaEvent_t ea = nullptr, eb = nullptr;
    if (pf && pf->timing) {
      ea = pf->next_event();
      eb = pf->next_event();
      if (ea) OKLS_CK(cudaEventRecord(ea, st));
    }
    OKLS_CK(launch_gemm(L, sms, st));
    if (pf) {
      if (ea && eb) {
        OKLS_CK(cudaEventRecord(eb, st));
        pf->recs.push_back({ea, eb, flops, g_in_ns, false});
      }
      if (L.total_tiles > 0) {
        pf->kernels += 1;
        pf->gemm_launches += 1;
        pf->gemm_flops += flops;
        if (g_in_ns) {
          pf->ns_launches += 1;
          pf->ns_flops += flops;
        }
      }
    }
    return OKLS_OK;
  }
};


void check_out(const Buf& b, int64_t rows, int64_t cols, int64_t batch, int64_t ld) {
  if (b.rows < rows || b.cols < cols || b.batch < batch || b.ld != ld || b.p == nullptr) g_plan_error = true;
}

void set_out16(GemmProblem& p, const Buf& hi, const Buf* hiT, const Buf* lo, const Buf* loT) {
  check_out(hi, p.rows, p.cols, p.batch, hi.ld);
  if (hiT) check_out(*hiT, p.cols, p.rows, p.batch, hi.ld);
  if (lo) check_out(*lo, p.rows, p.cols, p.batch, hi.ld);
  if (loT) check_out(*loT, p.cols, p.rows, p.batch, hi.ld);
  p.out_hi = hi.p;
  p.out_hi_t = hiT ? hiT->p : nullptr;
  p.out_lo = lo ? lo->p : nullptr;
  p.out_lo_t = loT ? loT->p : nullptr;
  p.ld16 = hi.ld;
  p.mat16 = hi.mat();
  p.split_out = lo ? 1 : 0;
}

// The GEMM stages of the coupled Newton-Schulz chain for 1 or 2 factors,
// handed to `sink` in order (one LaunchBuilder per stage: stage 0 is
// Y_1 = Y_0 T_0, then per iteration k >= 1 the T_k stage and the Y/Z stage).
// The stable order is kept: M_k = Z_k Y_k, Y_{k+1} = Y_k T_k,
// Z_{k+1} = T_k Z_k.  root_only: the last iteration forms only the square
// root (every factor must have root32), not P, its binary16 copy or their
// scales.  Each problem carries the counter slot of its factor (factor q's
// matrices use slots sum_{q' < q} batch_q' + b) for chain launches.  With a
// trace, the iterates of factor 0 are copied out between stages (per-stage
// launches only).
struct TraceOut {
  uint16_t* base = nullptr;  // [(3K+1)][count][d][d]
  int64_t count = 0, d = 0;
};

okls_status trace_copy(const TraceOut& tr, int slice, const Buf* b, cudaStream_t st) {
  if (!tr.base) return OKLS_OK;
  const int64_t dd = tr.d * tr.d;
  uint16_t* dst = tr.base + static_cast<int64_t>(slice) * tr.count * dd;
  if (!b) {
    OKLS_CK(cudaMemsetAsync(dst, 0, static_cast<size_t>(tr.count * dd * 2), st));
    return OKLS_OK;
  }
  OKLS_CK(cudaMemcpy2DAsync(dst, static_cast<size_t>(tr.d * 2), b->p, static_cast<size_t>(b->ld * 2),
                            static_cast<size_t>(tr.d * 2), static_cast<size_t>(tr.d * tr.count),
                            cudaMemcpyDeviceToDevice, st));
  return OKLS_OK;
}

template <class Sink>
okls_status ns_stages(Factor* const* fs, int nf, const Sched& sc, int split, float* scal, int scal_ld,
                      bool root_only, const TraceOut* tr, cudaStream_t st, Sink&& sink) {
  const int K = sc.iters;
  const int h = kHeadroom;
  int slot0[2] = {0, 0};
  for (int q = 1; q < nf; ++q) slot0[q] = slot0[q - 1] + fs[q - 1]->batch;
  okls_status s;
  // k = 0: Y_1 = Y_0 T_0 (Z_1 = T_0 written by the normaliser)
  {
    LaunchBuilder lb;
    const bool sp = split > 0, spo = split > 1;
    for (int q = 0; q < nf; ++q) {
      Factor& f = *fs[q];
      GemmProblem& p = lb.add(f.Y[0], f.T, sp, f.d, f.d, f.d, f.batch, EPI_NS_SCALE, false, true);
      set_out16(p, f.Y[1][0], nullptr, spo ? &f.Y[1][1] : nullptr, nullptr);
      p.alpha = std::ldexp(1.0f, -h);
      p.dep_slot = slot0[q];
    }
    if ((s = sink(lb)) != OKLS_OK) return s;
  }
  for (int k = 1; k < K; ++k) {
    const int cur = k & 1, nxt = cur ^ 1;
    const bool sp = split > k;       // operands of this iteration are pairs
    const bool spo = split > k + 1;  // outputs feed a split iteration
    {
      LaunchBuilder lb;  // T_k = a_k I + b_k Z_k Y_k
      for (int q = 0; q < nf; ++q) {
        Factor& f = *fs[q];
        GemmProblem& p = lb.add(f.Z[cur], f.Y[cur], sp, f.d, f.d, f.d, f.batch, EPI_NS_T, false, true);
        set_out16(p, f.T[0], nullptr, sp ? &f.T[1] : nullptr, nullptr);
        p.alpha = static_cast<float>(std::ldexp(sc.a[k], h));
        p.beta = static_cast<float>(std::ldexp(sc.b[k], sc.z[k] - h));
        p.dep_slot = slot0[q];
      }
      if ((s = sink(lb)) != OKLS_OK) return s;
    }
    if (tr && tr->base) {
      if ((s = trace_copy(*tr, 3 * k, &fs[0]->Y[cur][0], st)) != OKLS_OK) return s;
      if ((s = trace_copy(*tr, 3 * k + 1, &fs[0]->Z[cur][0], st)) != OKLS_OK) return s;
      if ((s = trace_copy(*tr, 3 * k + 2, &fs[0]->T[0], st)) != OKLS_OK) return s;
    }
    LaunchBuilder lb;
    for (int q = 0; q < nf; ++q) {
      Factor& f = *fs[q];
      if (k < K - 1) {
        GemmProblem& py = lb.add(f.Y[cur], f.T, sp, f.d, f.d, f.d, f.batch, EPI_NS_SCALE, false, true);
        set_out16(py, f.Y[nxt][0], nullptr, spo ? &f.Y[nxt][1] : nullptr, nullptr);
        py.alpha = std::ldexp(1.0f, -h);
        py.dep_slot = slot0[q];
        GemmProblem& pz = lb.add(f.T, f.Z[cur], sp, f.d, f.d, f.d, f.batch, EPI_NS_SCALE, false, true);
        set_out16(pz, f.Z[nxt][0], nullptr, spo ? &f.Z[nxt][1] : nullptr, nullptr);
        pz.alpha = std::ldexp(1.0f, sc.z[k] - sc.z[k + 1] - h);
        pz.dep_slot = slot0[q];
      } else {
        if (!root_only) {
          GemmProblem& pz = lb.add(f.T, f.Z[cur], sp, f.d, f.d, f.d, f.batch, EPI_NS_LAST, false, true);
          // in split mode the copy of P read by the X and whitening products
          // is a (hi, lo) pair as well
          set_out16(pz, f.Ph[0], nullptr, f.split ? &f.Ph[1] : nullptr, nullptr);
          pz.alpha = std::ldexp(1.0f, sc.z[k] - sc.z[k + 1] - h);
          pz.out32 = f.P32;
          pz.ld32 = f.d;
          pz.mat32 = static_cast<int64_t>(f.d) * f.d;
          pz.scal = scal;
          pz.scal_ld = scal_ld;
          pz.scal_slot = f.slot_pscale;
          pz.pi_slot = f.slot_pi;
          pz.cp_slot = f.slot_cprime;
          pz.pi_exp = sc.z[K] - h;
          pz.dep_slot = slot0[q];
        }
        if (f.root32) {
          GemmProblem& pr = lb.add(f.Y[cur], f.T, sp, f.d, f.d, f.d, f.batch, EPI_ROOT, false, true);
          pr.out32 = f.root32;
          pr.ld32 = f.d;
          pr.mat32 = static_cast<int64_t>(f.d) * f.d;
          pr.scal = scal;
          pr.scal_ld = scal_ld;
          pr.scal_slot = f.slot_rscale;
          pr.dep_slot = slot0[q];
        }
      }
    }
    if ((s = sink(lb)) != OKLS_OK) return s;
  }
  return OKLS_OK;
}

// A whole Newton-Schulz chain (its GEMM stages) as one persistent launch:
// the problem table and the completion counters live in the workspace; the
// table is built and uploaded once, when the handle is created (every
// pointer and constant in it is fixed for the handle's life).
struct ChainProgram {
  bool ready = false;
  GemmProblem* table = nullptr;  // device, kChainMaxProblems entries reserved
  uint32_t* done = nullptr;      // device, [stages][nslot]
  int nprob = 0, nstage = 0, nslot = 0;
  int64_t total_tiles = 0;
  double flops = 0.0;
};

constexpr int kChainMaxStages = 64;
// Chains run for factors of at most this size; past it the per-stage
// launches' fixed costs are small beside the products.
constexpr int kChainMaxD = 1024;

bool chain_enabled() {
  static const bool on = [] {
    const char* e = getenv("OKLS_NS_CHAIN");
    return !(e && e[0] == '0');
  }();
  return on;
}

size_t chain_table_bytes() { return static_cast<size_t>(kChainMaxProblems) * sizeof(GemmProblem); }
size_t chain_done_bytes(int nslot) { return static_cast<size_t>(kChainMaxStages) * nslot * 4; }

// Build the chain program of the GEMM stages for the factors `fs` and upload
// its table (synchronously; called when the handle is created).
okls_status build_chain(ChainProgram& cp, Factor* const* fs, int nf, const Sched& sc, int split, float* scal,
                        int scal_ld, bool root_only, int sms) {
  std::vector<GemmProblem> probs;
  std::vector<std::vector<int64_t>> need;  // per stage, per factor: completions of one matrix
  int stage = 0;
  int64_t base = 0;
  double flops = 0.0;
  okls_status s = ns_stages(fs, nf, sc, split, scal, scal_ld, root_only, nullptr, nullptr, [&](LaunchBuilder& lb) {
    double f = 0.0;
    okls_status s0 = lb.prepare(sms, base, &f);
    if (s0 != OKLS_OK) return s0;
    base = lb.L.total_tiles;
    flops += f;
    need.emplace_back(nf, 0);
    for (int i = 0; i < lb.L.nprob; ++i) {
      GemmProblem p = lb.L.prob[i];
      // factor index from the slot base
      int q = 0, acc = 0;
      for (; q < nf; ++q) {
        if (p.dep_slot == acc) break;
        acc += fs[q]->batch;
      }
      if (q == nf) return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: chain slot");
      p.stage = stage;
      p.dep_need = 0;
      if (stage > 0) {
        const int64_t nd = need[stage - 1][q];
        if (nd <= 0 || nd > 0x7fffffff) return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: chain dependency");
        p.dep_need = static_cast<int32_t>(nd);
      }
      need[stage][q] += 8 * p.tiles_per_mat;
      probs.push_back(p);
    }
    ++stage;
    return OKLS_OK;
  });
  if (s != OKLS_OK) return s;
  if (static_cast<int>(probs.size()) > kChainMaxProblems || stage > kChainMaxStages)
    return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: chain too long");
  int nslot = 0;
  for (int q = 0; q < nf; ++q) nslot += fs[q]->batch;
  if (nslot != cp.nslot) return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: chain slots");
  cp.nprob = static_cast<int>(probs.size());
  cp.nstage = stage;
  cp.total_tiles = base;
  cp.flops = flops;
  cudaError_t e = cudaMemcpy(cp.table, probs.data(), probs.size() * sizeof(GemmProblem), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(OKLS_ERR_CUDA, "chain table upload: %s", cudaGetErrorString(e));
  cp.ready = true;
  return OKLS_OK;
}

okls_status run_chain(const ChainProgram& cp, const CUtensorMap* maps, uint32_t* status, int sms, cudaStream_t st) {
  OKLS_CK(cudaMemsetAsync(cp.done, 0, static_cast<size_t>(cp.nstage) * cp.nslot * 4, st));
  ChainLaunch C;
  memset(&C, 0, sizeof(C));
  C.prob = cp.table;
  C.nprob = cp.nprob;
  C.nslot = cp.nslot;
  C.total_tiles = cp.total_tiles;
  C.done = cp.done;
  C.maps = maps;
  C.status = status;
  C.wait_cycles = g_wait.cycles;
  C.unloaded_tile = g_wait.unloaded_tile;
  Prof* pf = g_prof;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (pf && pf->timing) {
    ea = pf->next_event();
    eb = pf->next_event();
    if (ea) OKLS_CK(cudaEventRecord(ea, st));
  }
  OKLS_CK(launch_chain(C, sms, st));
  if (pf) {
    if (ea && eb) {
      OKLS_CK(cudaEventRecord(eb, st));
      pf->recs.push_back({ea, eb, cp.flops, true, false});
    }
    pf->kernels += 1;
    pf->gemm_launches += 1;
    pf->gemm_flops += cp.flops;
    pf->ns_launches += 1;
    pf->ns_flops += cp.flops;
  }
  return OKLS_OK;
}

// Normalisation of the factors (k_normalise: Y_0, T_0, Z_1 and, for a
// factor-product output, S's mirrored lower triangle).
okls_status ns_normalise(Factor* const* fs, int nf, const Sched& sc, int split, float ridge, float* scal,
                         int scal_ld, uint32_t* status, cudaStream_t st) {
  for (int q = 0; q < nf; ++q) {
    Factor& f = *fs[q];
    NormaliseArgs A;
    memset(&A, 0, sizeof(A));
    A.S = f.S;
    A.upper_only = f.S_upper_only ? 1 : 0;
    A.d = f.d;
    A.ld16 = f.Y[0][0].ld;
    A.mat16 = f.Y[0][0].mat();
    A.Y = f.Y[0][0].p;
    A.T = f.T[0].p;
    A.Z = f.Z[1][0].p;
    A.split_y = split > 0;
    A.split_t = split > 0;
    A.split_z = split > 1;
    if (A.split_y) {
      A.Ylo = f.Y[0][1].p;
      A.Tlo = f.T[1].p;
    }
    if (A.split_z) A.Zlo = f.Z[1][1].p;
    A.a0 = static_cast<float>(sc.a[0]);
    A.b0 = static_cast<float>(sc.b[0]);
    A.z1 = sc.z[1];
    A.ridge = ridge;
    A.scal = scal;
    A.scal_ld = scal_ld;
    A.slot_cprime = f.slot_cprime;
    A.slot_sumsq = f.slot_sumsq;
    A.status = status;
    // per element: the upper triangle of S read and its mirror written
    // (upper-only input) or all of S read (full input); Y_0, T_0, Z_1 (and
    // low halves) written
    const double per = 4.0 + 6.0 + 2.0 * (A.split_y + A.split_t + A.split_z);
    okls_status s0 = bw_launch(per * f.batch * static_cast<double>(f.d) * f.d, st,
                               [&] { return launch_normalise(A, f.batch, st); });
    if (s0 != OKLS_OK) return s0;
  }
  return OKLS_OK;
}

// Factors with d <= 128 run the whole chain in one fused on-chip kernel
// (plain binary16 mode); OKLS_NS_SMALL=0 sends them through the general path.
constexpr int kSmallMaxD = 128;
bool small_enabled() {
  static const bool on = [] {
    const char* e = getenv("OKLS_NS_SMALL");
    return !(e && e[0] == '0');
  }();
  return on;
}

bool takes_small(const Factor& f, int split) { return split == 0 && small_enabled() && f.d <= kSmallMaxD; }

okls_status run_ns_small(Factor* const* fs, int nf, const Sched& sc, float ridge, float* scal, int scal_ld,
                         uint32_t* status, cudaStream_t st, const TraceOut* tr, bool root_only) {
  SmallNsArgs A;
  memset(&A, 0, sizeof(A));
  A.nf = nf;
  double flops = 0.0;
  for (int q = 0; q < nf; ++q) {
    const Factor& f = *fs[q];
    SmallNsFactor& g = A.f[q];
    g.S = f.S;
    g.upper_only = f.S_upper_only ? 1 : 0;
    g.d = f.d;
    g.count = f.batch;
    g.P32 = f.P32;
    g.Ph = f.Ph[0].p;
    g.ph_ld = f.Ph[0].ld;
    g.ph_mat = f.Ph[0].mat();
    g.root32 = f.root32;
    g.slot_sumsq = f.slot_sumsq;
    g.slot_cprime = f.slot_cprime;
    g.slot_pscale = f.slot_pscale;
    g.slot_rscale = f.slot_rscale;
    g.slot_pi = f.slot_pi;
    // algorithmic work of the chain: 27 (or 28 with the root) d^3 products
    flops += 2.0 * f.d * static_cast<double>(f.d) * f.d * f.batch * (3.0 * sc.iters - 3.0 + (f.root32 ? 1.0 : 0.0));
  }
  A.scal = scal;
  A.scal_ld = scal_ld;
  A.ridge = ridge;
  A.iters = sc.iters;
  for (int k = 0; k < sc.iters; ++k) {
    A.a[k] = static_cast<float>(sc.a[k]);
    A.b[k] = static_cast<float>(sc.b[k]);
  }
  for (int k = 0; k <= sc.iters; ++k) A.z[k] = sc.z[k];
  A.want_p = root_only ? 0 : 1;
  A.trace = (tr && tr->base) ? tr->base : nullptr;
  A.trace_count = tr ? tr->count : 0;
  A.status = status;
  Prof* pf = g_prof;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (pf && pf->timing) {
    ea = pf->next_event();
    eb = pf->next_event();
    if (ea) OKLS_CK(cudaEventRecord(ea, st));
  }
  OKLS_CK(launch_ns_small(A, st));
  if (pf) {
    if (ea && eb) {
      OKLS_CK(cudaEventRecord(eb, st));
      pf->recs.push_back({ea, eb, flops, true, false});
    }
    pf->kernels += 1;
    pf->gemm_launches += 1;
    pf->gemm_flops += flops;
    pf->ns_launches += 1;
    pf->ns_flops += flops;
  }
  return OKLS_OK;
}

// Normalisation and the Newton-Schulz chain of 1 or 2 factors: factors with
// d <= 128 (plain mode) in the fused kernel, the rest as one chain launch when
// `chain` holds their program, else as one launch per stage.  A trace is
// taken from factor 0 only, so a traced run keeps factor 0 on one path.
okls_status run_ns(Factor* const* fs, int nf, const Sched& sc, int split, float ridge, float* scal,
                   int scal_ld, const CUtensorMap* maps, uint32_t* status, int sms, cudaStream_t st,
                   const TraceOut* tr, bool root_only = false, const ChainProgram* chain = nullptr) {
  for (int q = 0; q < nf && root_only; ++q)
    if (!fs[q]->root32) return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: square-root output");
  if (sc.iters > kSmallMaxIters) return fail(OKLS_ERR_UNSUPPORTED, "more than %d Newton-Schulz steps", kSmallMaxIters);
  Factor* small[2];
  Factor* big[2];
  int ns = 0, nb = 0;
  for (int q = 0; q < nf; ++q) {
    if (takes_small(*fs[q], split))
      small[ns++] = fs[q];
    else
      big[nb++] = fs[q];
  }
  okls_status s = OKLS_OK;
  if (ns > 0) {
    const bool tr_small = tr && tr->base && small[0] == fs[0];
    if ((s = run_ns_small(small, ns, sc, ridge, scal, scal_ld, status, st, tr_small ? tr : nullptr, root_only)) !=
        OKLS_OK)
      return s;
  }
  if (nb == 0) return OKLS_OK;
  const bool tr_big = tr && tr->base && big[0] == fs[0];
  if ((s = ns_normalise(big, nb, sc, split, ridge, scal, scal_ld, status, st)) != OKLS_OK) return s;
  if (chain && chain->ready && !tr_big) return run_chain(*chain, maps, status, sms, st);
  if (tr_big) {
    if ((s = trace_copy(*tr, 0, &big[0]->Y[0][0], st)) != OKLS_OK) return s;
    if ((s = trace_copy(*tr, 1, nullptr, st)) != OKLS_OK) return s;
    if ((s = trace_copy(*tr, 2, &big[0]->T[0], st)) != OKLS_OK) return s;
  }
  g_in_ns = true;
  s = ns_stages(big, nb, sc, split, scal, scal_ld, root_only, tr_big ? tr : nullptr, st,
                [&](LaunchBuilder& lb) { return lb.go(maps, status, sms, st); });
  g_in_ns = false;
  if (s != OKLS_OK) return s;
  if (tr_big && !root_only) return trace_copy(*tr, 3 * sc.iters, &big[0]->Ph[0], st);
  return OKLS_OK;
}

}  // namespace

// ====================================================================== handle
struct okls_handle_s {
  okls_config cfg;
  int sms = 0;
  Sched sched;
  float *M = nullptr, *Sa = nullptr, *Sb = nullptr, *Pa = nullptr, *Pb = nullptr;
  Factor fa, fb;
  Buf Gh, GhT, Nh, Xb, XaT;  // Ghat (m x n), Ghat^T (n x m), Nhat (m x n), X_b / Q (m x n), X_a^T (n x m)
  float *sq_a = nullptr, *sq_b = nullptr;  // Shampoo: fp32 square roots L^1/2, R^1/2 between the chains
  float* V = nullptr;                      // SOAP: second moment in the eigenbasis; Clean: Main block's
  // Clean: block moments of A (m x r), B (r x n), pooled second moments, and
  // the refreshed bases of a refresh step (workspace)
  float *MA = nullptr, *MB = nullptr, *vA = nullptr, *vB = nullptr, *vC = nullptr;
  float *ULn = nullptr, *URn = nullptr, *lamLn = nullptr, *lamRn = nullptr;
  bool soap_large = false;   // SOAP past one CTA's shared memory (batched fp32 GEMMs)
  SoapLarge sl;
  bool clean_large = false;  // Clean past one CTA's shared memory (batched fp32 GEMMs)
  ClLarge cl;                // its buffers (the state pointers above, plus workspace)
  float* scal = nullptr;
  uint32_t* status = nullptr;
  CUtensorMap* maps = nullptr;
  std::vector<int> boxes;  // box rows of each descriptor in the table
  float *part_g = nullptr, *part_a = nullptr, *part_b = nullptr;  // fixed-slot partial sums
  int64_t part_g_ld = 0, part_a_ld = 0, part_b_ld = 0;
  int64_t t = 0;
  Prof prof;
  WaitSetting wait;  // okls_set_wait_limit
  // Newton-Schulz chains as single persistent launches (factors up to
  // kChainMaxD): OKLS uses chain[0]; Shampoo chain[0] (square roots) and
  // chain[1] (inverse square roots of those)
  ChainProgram chain[2];
  int nchain = 0;
};

namespace {

struct Layout {
  size_t state_bytes = 0, ws_bytes = 0;
};

// SOAP runs one CTA per matrix up to 128 x 128; past that (to 544), or with
// OKLS_SOAP_LARGE=1, the batched-GEMM path.
bool soap_large_path(const okls_config& c) {
  const char* e = getenv("OKLS_SOAP_LARGE");
  if (e && e[0] == '1') return true;
  return c.m > 128 || c.n > 128;
}

// A SOAP side's refresh runs the blocked Jacobi solver past the logged-rotation
// solver's range, or past 128 with OKLS_SOAP_BLOCKED=1 (tests run the blocked
// solver at sizes the oracle finishes quickly).
bool soap_blocked_side(int64_t d) {
  if (d > kClMaxK) return true;
  const char* e = getenv("OKLS_SOAP_BLOCKED");
  return e && e[0] == '1' && d > 128;
}

// Clean runs one CTA per factor while a factor's panels fit its shared
// memory (m, n <= 128, r + p <= 64); past that, or with OKLS_CLEAN_LARGE=1,
// the batched-GEMM path.
bool clean_large_path(const okls_config& c) {
  const char* e = getenv("OKLS_CLEAN_LARGE");
  if (e && e[0] == '1') return true;
  return c.m > 128 || c.n > 128 || c.rank + c.oversample > 64;
}

// Clean: bases U_L (m x r), U_R (n x r) and eigenvalues in P_a / P_b and
// S_a / S_b, Main moments in M / V, the A and B block moments and the pooled
// second moments; the workspace holds the status word and a refresh's output.
okls_status plan_clean(const okls_config& c, uint8_t* state, uint8_t* ws, okls_handle_s* h, Layout* out) {
  const int64_t B = c.batch, m = c.m, n = c.n, r = c.rank;
  Planner sp;
  sp.base = state;
  auto f32 = [](Planner& pl, int64_t elems) { return static_cast<float*>(pl.take(static_cast<size_t>(elems * 4))); };
  float* UL = f32(sp, B * m * r);
  float* UR = f32(sp, B * n * r);
  float* lamL = f32(sp, B * r);
  float* lamR = f32(sp, B * r);
  float* M = f32(sp, B * r * r);
  float* V = f32(sp, B * r * r);
  float* MA = f32(sp, B * m * r);
  float* MB = f32(sp, B * r * n);
  float* vA = f32(sp, B * r);
  float* vB = f32(sp, B * r);
  float* vC = f32(sp, B);
  Planner wp;
  wp.base = ws;
  uint32_t* status = static_cast<uint32_t*>(wp.take(256));
  float* ULn = f32(wp, B * m * r);
  float* URn = f32(wp, B * n * r);
  float* lamLn = f32(wp, B * r);
  float* lamRn = f32(wp, B * r);
  const bool large = clean_large_path(c);
  ClLarge cl;
  memset(&cl, 0, sizeof(cl));
  if (large) {
    const int64_t k = static_cast<int64_t>(c.rank) + c.oversample, dmax = m > n ? m : n;
    cl.Om = f32(wp, B * dmax * k);
    cl.Y = f32(wp, B * dmax * k);
    cl.X = f32(wp, B * dmax * k);
    cl.T1 = f32(wp, B * dmax * k);
    cl.Gram = f32(wp, B * k * k);
    cl.Rinv = f32(wp, B * k * k);
    cl.WU = f32(wp, B * k * r);
    cl.P = f32(wp, B * k * r);
    cl.nu = f32(wp, B);
    cl.Mn = f32(wp, B * r * r);
    cl.Sm = f32(wp, B * r * r);
    cl.MAn = f32(wp, B * m * r);
    cl.MBn = f32(wp, B * r * n);
    cl.vAn = f32(wp, B * r);
    cl.vBn = f32(wp, B * r);
    cl.GU = f32(wp, B * m * r);
    cl.UG = f32(wp, B * r * n);
    cl.S = f32(wp, B * r * r);
    cl.Nm = f32(wp, B * r * r);
    cl.Cb = f32(wp, B * m * n);
    cl.part = f32(wp, B * kClParts);
    cl.cden = f32(wp, B);
    cl.KK = k > 128 ? f32(wp, B * std::max<int64_t>(2 * (k + 1) * (k + 1),
                                                   static_cast<int64_t>(eig_scratch_floats(static_cast<int>(k)))))
                    : nullptr;
  }
  out->state_bytes = sp.off;
  out->ws_bytes = wp.off;
  if (h) {
    h->Pa = UL;
    h->Pb = UR;
    h->Sa = lamL;
    h->Sb = lamR;
    h->M = M;
    h->V = V;
    h->MA = MA;
    h->MB = MB;
    h->vA = vA;
    h->vB = vB;
    h->vC = vC;
    h->ULn = ULn;
    h->URn = URn;
    h->lamLn = lamLn;
    h->lamRn = lamRn;
    h->status = status;
    h->clean_large = large;
    if (large) {
      cl.batch = static_cast<int>(B);
      cl.m = static_cast<int>(m);
      cl.n = static_cast<int>(n);
      cl.r = c.rank;
      cl.p = c.oversample;
      cl.q = c.power_iters;
      cl.k = c.rank + c.oversample;
      cl.status = status;
      cl.UL = UL;
      cl.UR = UR;
      cl.lamL = lamL;
      cl.lamR = lamR;
      cl.M = M;
      cl.V = V;
      cl.MA = MA;
      cl.MB = MB;
      cl.vA = vA;
      cl.vB = vB;
      cl.vC = vC;
      cl.ULn = ULn;
      cl.URn = URn;
      cl.lamLn = lamLn;
      cl.lamRn = lamRn;
      h->cl = cl;
    }
  }
  return OKLS_OK;
}

// Lays out state and workspace; with bases set, fills the handle too.
// A step's Newton-Schulz GEMM stages run as one chain launch when every
// factor that does not take the fused small kernel has d <= kChainMaxD
// (OKLS_NS_CHAIN=0: always one launch per stage).
bool chain_eligible(const okls_config& c) {
  if (!chain_enabled()) return false;
  if (c.method != OKLS_METHOD_OKLS && c.method != OKLS_METHOD_SHAMPOO) return false;
  const int split = c.ns_split_iters;
  bool any = false;
  for (int64_t d : {c.m, c.n}) {
    if (split == 0 && small_enabled() && d <= kSmallMaxD) continue;
    if (d > kChainMaxD) return false;
    any = true;
  }
  return any;
}

// counter slots of a step's chain: the batch of each factor that runs in it
int chain_slots(const okls_config& c) {
  int n = 0;
  for (int64_t d : {c.m, c.n})
    if (!(c.ns_split_iters == 0 && small_enabled() && d <= kSmallMaxD)) n += static_cast<int>(c.batch);
  return n;
}

okls_status plan(const okls_config& c, uint8_t* state, uint8_t* ws, okls_handle_s* h, Layout* out) {
  const int64_t B = c.batch, m = c.m, n = c.n;
  if (c.method == OKLS_METHOD_CLEAN) return plan_clean(c, state, ws, h, out);
  Planner sp;
  sp.base = state;
  float* M = static_cast<float*>(sp.take(static_cast<size_t>(B * m * n * 4)));
  float* Sa = static_cast<float*>(sp.take(static_cast<size_t>(B * m * m * 4)));
  float* Sb = static_cast<float*>(sp.take(static_cast<size_t>(B * n * n * 4)));
  float* Pa = static_cast<float*>(sp.take(static_cast<size_t>(B * m * m * 4)));
  float* Pb = static_cast<float*>(sp.take(static_cast<size_t>(B * n * n * 4)));
  const bool soap = c.method == OKLS_METHOD_SOAP;
  float* V = soap ? static_cast<float*>(sp.take(static_cast<size_t>(B * m * n * 4))) : nullptr;
  Planner wp;
  wp.base = ws;
  CUtensorMap* maps = static_cast<CUtensorMap*>(wp.take(kMapTableBytes, 128));
  float* scal = static_cast<float*>(wp.take(static_cast<size_t>(SC_COUNT * B * 4)));
  uint32_t* status = static_cast<uint32_t*>(wp.take(256));
  if (soap) {
    // SOAP keeps everything in the state; the workspace holds the status word
    // (and, past one CTA, the batched path's buffers)
    const bool large = soap_large_path(c);
    SoapLarge sl;
    memset(&sl, 0, sizeof(sl));
    if (large) {
      const int64_t dmax = m > n ? m : n;
      const int64_t big = std::max(m * n, dmax * dmax);
      auto f32 = [&](int64_t elems) { return static_cast<float*>(wp.take(static_cast<size_t>(elems * 4))); };
      sl.Gf = f32(B * m * n);
      sl.Gp = f32(B * m * n);
      sl.Mp = f32(B * m * n);
      sl.T = f32(B * big);
      for (int side = 0; side < 2; ++side) {
        const int64_t d = side == 0 ? m : n;
        SoapSideBufs& sb = side == 0 ? sl.sideL : sl.sideR;
        sb.blocked = soap_blocked_side(d) ? 1 : 0;
        sb.Qh = f32(B * d * d);
        sb.A = f32(B * d * d);
        sb.P = f32(B * d * d);
        if (sb.blocked) {
          sb.BJ = f32(B * static_cast<int64_t>(bj_scratch_floats(static_cast<int>(d))));
        } else {
          sb.Wq = f32(B * d * d);
          if (d > 128) sb.KK = f32(B * static_cast<int64_t>(eig_scratch_floats(static_cast<int>(d))));
        }
      }
    }
    out->state_bytes = sp.off;
    out->ws_bytes = wp.off;
    if (h) {
      h->M = M;
      h->Sa = Sa;
      h->Sb = Sb;
      h->Pa = Pa;
      h->Pb = Pb;
      h->V = V;
      h->scal = scal;
      h->status = status;
      h->maps = maps;
      h->soap_large = large;
      if (large) {
        sl.batch = static_cast<int>(B);
        sl.m = static_cast<int>(m);
        sl.n = static_cast<int>(n);
        sl.M = M;
        sl.V = V;
        sl.L = Sa;
        sl.R = Sb;
        sl.QL = Pa;
        sl.QR = Pb;
        sl.status = status;
        h->sl = sl;
      }
    }
    return OKLS_OK;
  }
  const int64_t pg_ld = kMaxStatParts, pa_ld = factor_parts(m), pb_ld = factor_parts(n);
  float* part_g = static_cast<float*>(wp.take(static_cast<size_t>(2 * B * pg_ld * 4)));
  float* part_a = static_cast<float*>(wp.take(static_cast<size_t>(B * pa_ld * 4)));
  float* part_b = static_cast<float*>(wp.take(static_cast<size_t>(B * pb_ld * 4)));
  const bool shampoo = c.method == OKLS_METHOD_SHAMPOO;
  // Shampoo has no momentum (N = G) and no preconditioned factor inputs, so
  // Nhat and X_a^T are not needed; it keeps each factor's square root instead
  Buf Gh = wp.buf16(m, n, B), GhT = wp.buf16(n, m, B);
  Buf Nh = shampoo ? Buf() : wp.buf16(m, n, B);
  Buf Xb = wp.buf16(m, n, B);
  Buf XaT = shampoo ? Buf() : wp.buf16(n, m, B);
  float* sq_a = shampoo ? static_cast<float*>(wp.take(static_cast<size_t>(B * m * m * 4))) : nullptr;
  float* sq_b = shampoo ? static_cast<float*>(wp.take(static_cast<size_t>(B * n * n * 4))) : nullptr;
  Factor fa, fb;
  const bool split = c.ns_split_iters > 0;
  plan_factor(wp, fa, static_cast<int>(m), static_cast<int>(B), split);
  plan_factor(wp, fb, static_cast<int>(n), static_cast<int>(B), split);
  // chain programs: the problem tables and completion counters
  const int nchain = chain_eligible(c) ? (shampoo ? 2 : 1) : 0;
  ChainProgram chains[2];
  for (int i = 0; i < nchain; ++i) {
    chains[i].nslot = chain_slots(c);
    chains[i].table = static_cast<GemmProblem*>(wp.take(chain_table_bytes()));
    chains[i].done = static_cast<uint32_t*>(wp.take(chain_done_bytes(chains[i].nslot)));
  }
  if (wp.err != OKLS_OK) return wp.err;
  out->state_bytes = sp.off;
  out->ws_bytes = wp.off;
  if (h) {
    h->M = M;
    h->Sa = Sa;
    h->Sb = Sb;
    h->Pa = Pa;
    h->Pb = Pb;
    fa.S = Sa;
    fa.S_upper_only = true;
    fa.P32 = Pa;
    fa.slot_sumsq = SC_SUMSQ_SA;
    fa.slot_cprime = SC_CPRIME_A;
    fa.slot_pi = SC_PI_A;
    fa.slot_pscale = SC_PSCALE_A;
    fa.slot_rscale = SC_RSCALE_A;
    fb.S = Sb;
    fb.S_upper_only = true;
    fb.P32 = Pb;
    fb.slot_sumsq = SC_SUMSQ_SB;
    fb.slot_cprime = SC_CPRIME_B;
    fb.slot_pi = SC_PI_B;
    fb.slot_pscale = SC_PSCALE_B;
    fb.slot_rscale = SC_RSCALE_B;
    h->fa = fa;
    h->fb = fb;
    h->Gh = Gh;
    h->GhT = GhT;
    h->Nh = Nh;
    h->Xb = Xb;
    h->XaT = XaT;
    h->sq_a = sq_a;
    h->sq_b = sq_b;
    h->scal = scal;
    h->status = status;
    h->maps = maps;
    h->part_g = part_g;
    h->part_a = part_a;
    h->part_b = part_b;
    h->part_g_ld = pg_ld;
    h->part_a_ld = pa_ld;
    h->part_b_ld = pb_ld;
    h->boxes = wp.boxes;
    h->nchain = nchain;
    for (int i = 0; i < nchain; ++i) h->chain[i] = chains[i];
    // upload the descriptor table once
    if (!wp.maps.empty()) {
      cudaError_t e = cudaMemcpy(maps, wp.maps.data(), wp.maps.size() * sizeof(CUtensorMap),
                                 cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return fail(OKLS_ERR_CUDA, "descriptor upload: %s", cudaGetErrorString(e));
    }
  }
  return OKLS_OK;
}

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.0f; }

okls_status validate(const okls_config* c) {
  if (!c) return fail(OKLS_ERR_INVALID_ARG, "config is NULL");
  if (c->batch < 1 || c->m < 1 || c->n < 1)
    return fail(OKLS_ERR_INVALID_ARG, "batch, m, n must be >= 1 (got %lld, %lld, %lld)",
                static_cast<long long>(c->batch), static_cast<long long>(c->m), static_cast<long long>(c->n));
  if (c->m > 32768 || c->n > 32768 || c->batch > 65535)
    return fail(OKLS_ERR_UNSUPPORTED, "m, n <= 32768 and batch <= 65535 supported");
  if (c->param_dtype != OKLS_F32 && c->param_dtype != OKLS_BF16)
    return fail(OKLS_ERR_INVALID_ARG, "param_dtype %d", c->param_dtype);
  if (c->grad_dtype != OKLS_F32 && c->grad_dtype != OKLS_BF16)
    return fail(OKLS_ERR_INVALID_ARG, "grad_dtype %d", c->grad_dtype);
  if (!(c->lr_peak > 0.0f) || !std::isfinite(c->lr_peak)) return fail(OKLS_ERR_INVALID_ARG, "lr_peak must be > 0");
  if (!(c->beta1 >= 0.0f && c->beta1 < 1.0f)) return fail(OKLS_ERR_INVALID_ARG, "beta1 must be in [0, 1)");
  if (!(c->beta2 >= 0.0f && c->beta2 < 1.0f)) return fail(OKLS_ERR_INVALID_ARG, "beta2 must be in [0, 1)");
  if (!finite_nonneg(c->eps)) return fail(OKLS_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!finite_nonneg(c->weight_decay)) return fail(OKLS_ERR_INVALID_ARG, "weight_decay must be >= 0");
  if (c->ns_iters < 2 || c->ns_iters > 32) return fail(OKLS_ERR_INVALID_ARG, "ns_iters must be in [2, 32]");
  if (c->ns_split_iters < 0 || c->ns_split_iters > c->ns_iters)
    return fail(OKLS_ERR_INVALID_ARG, "ns_split_iters must be in [0, ns_iters]");
  if (!(c->ns_lo > 0.0f && c->ns_lo < 1.0f)) return fail(OKLS_ERR_INVALID_ARG, "ns_lo must be in (0, 1)");
  if (!finite_nonneg(c->ridge)) return fail(OKLS_ERR_INVALID_ARG, "ridge must be finite and >= 0");
  if (c->root_every < 0) return fail(OKLS_ERR_INVALID_ARG, "root_every must be >= 0 (0 means 1)");
  if (c->method != OKLS_METHOD_OKLS && c->method != OKLS_METHOD_SHAMPOO && c->method != OKLS_METHOD_SOAP &&
      c->method != OKLS_METHOD_CLEAN)
    return fail(OKLS_ERR_INVALID_ARG, "method %d", c->method);
  if (c->method == OKLS_METHOD_CLEAN) {
    if (c->rank < 1 || c->oversample < 0 || c->power_iters < 0 || c->power_iters > 16)
      return fail(OKLS_ERR_INVALID_ARG, "Clean needs rank >= 1, oversample >= 0, power_iters in [0, 16]");
    const int64_t k = static_cast<int64_t>(c->rank) + c->oversample;
    if (k > c->m || k > c->n)
      return fail(OKLS_ERR_INVALID_ARG, "rank + oversample (%lld) exceeds min(m, n)", static_cast<long long>(k));
    if (c->m > 16384 || c->n > 16384 || k > kClMaxK)
      return fail(OKLS_ERR_UNSUPPORTED, "Clean runs for m, n <= 16384 and rank + oversample <= %d in this build",
                  kClMaxK);
  } else if (c->rank != 0 || c->oversample != 0 || c->power_iters != 0) {
    return fail(OKLS_ERR_INVALID_ARG, "rank, oversample and power_iters are Clean's; leave them zero");
  }
  if (c->method == OKLS_METHOD_SOAP && (c->m > kSoapLargeMax || c->n > kSoapLargeMax))
    return fail(OKLS_ERR_UNSUPPORTED, "SOAP runs for m, n <= %d in this build; got %lld x %lld", kSoapLargeMax,
                static_cast<long long>(c->m), static_cast<long long>(c->n));
  for (int i = 0; i < 3; ++i)
    if (c->reserved[i] != 0) return fail(OKLS_ERR_INVALID_ARG, "reserved fields must be zero");
  return OKLS_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SOAP (Clean page, Appendix C, Algorithm 4): the step, then the eigenbasis
// refresh after steps t with t % root_every == 0.
okls_status soap_step(okls_handle_s* h, void* W, const void* G, float lr, cudaStream_t st) {
  const okls_config& c = h->cfg;
  const int64_t t1 = h->t + 1;
  ProfScope scope(&h->prof);
  SoapArgs A;
  memset(&A, 0, sizeof(A));
  A.batch = static_cast<int>(c.batch);
  A.m = static_cast<int>(c.m);
  A.n = static_cast<int>(c.n);
  A.G = G;
  A.W = W;
  A.g_bf16 = c.grad_dtype == OKLS_BF16;
  A.w_bf16 = c.param_dtype == OKLS_BF16;
  A.M = h->M;
  A.V = h->V;
  A.L = h->Sa;
  A.R = h->Sb;
  A.QL = h->Pa;
  A.QR = h->Pb;
  A.beta1 = c.beta1;
  A.beta2 = c.beta2;
  A.eps = c.eps;
  A.lr = lr;
  A.decay = static_cast<float>(1.0 - static_cast<double>(lr) * c.weight_decay * (static_cast<double>(lr) / c.lr_peak));
  A.bc1 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(c.beta1), static_cast<double>(t1))));
  A.bc2 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(c.beta2), static_cast<double>(t1))));
  A.status = h->status;
  const int64_t every = c.root_every > 1 ? c.root_every : 1;
  if (h->soap_large) {
    SoapLarge S = h->sl;
    S.G = G;
    S.W = W;
    S.g_bf16 = A.g_bf16;
    S.w_bf16 = A.w_bf16;
    S.beta1 = A.beta1;
    S.beta2 = A.beta2;
    S.eps = A.eps;
    S.lr = A.lr;
    S.decay = A.decay;
    S.bc1 = A.bc1;
    S.bc2 = A.bc2;
    S.max_sweeps = 15;
    // one rule for the sides solved together; a blocked side takes its own
    S.tol2 = soap_tol2(std::max(c.m, c.n));
    int launches = 0;
    OKLS_CK(soap_large_step(S, t1 % every == 0, st, &launches));
    note_kernels(launches);
    h->t = t1;
    return OKLS_OK;
  }
  OKLS_CK(launch_soap_step(A, st));
  note_kernels(1);
  if (t1 % every == 0) {
    SoapRefreshArgs R;
    memset(&R, 0, sizeof(R));
    R.count = static_cast<int>(c.batch);
    R.S0 = h->Sa;
    R.S1 = h->Sb;
    R.Q0 = h->Pa;
    R.Q1 = h->Pb;
    R.d0 = static_cast<int>(c.m);
    R.d1 = static_cast<int>(c.n);
    // Jacobi converges quadratically; 1e-6 relative off-diagonal is the
    // fp32 floor for these sizes
    R.max_sweeps = 15;
    R.tol2 = 1e-12f;
    R.status = h->status;
    OKLS_CK(launch_soap_refresh(R, st));
    note_kernels(1);
  }
  h->t = t1;
  return OKLS_OK;
}

CleanArgs clean_args(okls_handle_s* h) {
  const okls_config& c = h->cfg;
  CleanArgs A;
  memset(&A, 0, sizeof(A));
  A.batch = static_cast<int>(c.batch);
  A.m = static_cast<int>(c.m);
  A.n = static_cast<int>(c.n);
  A.r = c.rank;
  A.p = c.oversample;
  A.q = c.power_iters;
  A.UL = h->Pa;
  A.UR = h->Pb;
  A.lamL = h->Sa;
  A.lamR = h->Sb;
  A.ULn = h->ULn;
  A.URn = h->URn;
  A.lamLn = h->lamLn;
  A.lamRn = h->lamRn;
  A.Mm = h->M;
  A.Vm = h->V;
  A.MA = h->MA;
  A.MB = h->MB;
  A.vA = h->vA;
  A.vB = h->vB;
  A.vC = h->vC;
  A.status = h->status;
  return A;
}

// Clean (Algorithm 1 of the Clean page): at steps t with (t - 1) % T == 0
// (T = root_every) both factors are re-sketched (Algorithm 3) and the moments
// moved to the new bases (Eqns. (14)-(15)); then the block step of
// Eqns. (10)-(13) and (16) with alpha = 1.
okls_status clean_step(okls_handle_s* h, void* W, const void* G, float lr, const float* noise, cudaStream_t st) {
  const okls_config& c = h->cfg;
  const int64_t t1 = h->t + 1;
  const int64_t every = c.root_every > 1 ? c.root_every : 1;
  const bool refresh = (t1 - 1) % every == 0;
  if (refresh && !noise) return fail(OKLS_ERR_INVALID_ARG, "step %lld refreshes the sketch: noise is required",
                                     static_cast<long long>(t1));
  if (noise && !aligned(noise, 16)) return fail(OKLS_ERR_UNSUPPORTED, "noise must be 16-byte aligned");
  ProfScope scope(&h->prof);
  CleanArgs A = clean_args(h);
  A.G = G;
  A.W = W;
  A.g_bf16 = c.grad_dtype == OKLS_BF16;
  A.w_bf16 = c.param_dtype == OKLS_BF16;
  A.noise = noise;
  A.warm = h->t > 0;
  A.beta1 = c.beta1;
  A.beta2 = c.beta2;
  A.eps = c.eps;
  A.alr = lr;
  A.decay = static_cast<float>(1.0 - static_cast<double>(lr) * c.weight_decay * (static_cast<double>(lr) / c.lr_peak));
  A.bc1 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(c.beta1), static_cast<double>(t1))));
  A.bc2 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(c.beta2), static_cast<double>(t1))));
  // Jacobi converges quadratically; 1e-6 relative off-diagonal is the fp32
  // floor up to 128 columns, and that floor grows like sqrt(k) past it
  A.max_sweeps = 15;
  A.tol2 = 1e-12f * std::max(1.0f, static_cast<float>(c.rank + c.oversample) / 128.0f);
  if (h->clean_large) {
    ClLarge L = h->cl;
    L.warm = A.warm;
    L.beta1 = A.beta1;
    L.beta2 = A.beta2;
    L.eps = A.eps;
    L.alr = A.alr;
    L.decay = A.decay;
    L.bc1 = A.bc1;
    L.bc2 = A.bc2;
    L.max_sweeps = A.max_sweeps;
    L.tol2 = A.tol2;
    L.G = G;
    L.W = W;
    L.g_bf16 = A.g_bf16;
    L.w_bf16 = A.w_bf16;
    L.noise = noise;
    int launches = 0;
    if (refresh) OKLS_CK(clean_large_refresh(L, st, &launches));
    OKLS_CK(clean_large_step(L, st, &launches));
    note_kernels(launches);
    h->t = t1;
    return OKLS_OK;
  }
  if (refresh) {
    OKLS_CK(launch_clean_refresh(A, st));
    note_kernels(2);
  }
  OKLS_CK(launch_clean_step(A, st));
  note_kernels(1);
  h->t = t1;
  return OKLS_OK;
}

okls_status step_impl(okls_handle h, void* W, const void* G, float lr, const float* noise, void* stream);

// The factors of a step's chain: those that do not take the fused small
// kernel, in the order run_ns hands them on.
int chain_factor_list(Factor* const* fs, int nf, int split, Factor** out) {
  int n = 0;
  for (int q = 0; q < nf; ++q)
    if (!takes_small(*fs[q], split)) out[n++] = fs[q];
  return n;
}

// Build the handle's chain programs (once, at creation): the same factor
// set-ups as the step's run_ns calls.
okls_status build_chains(okls_handle_s* h) {
  const okls_config& c = h->cfg;
  BoxScope boxes(&h->boxes);
  const int sld = static_cast<int>(c.batch);
  Factor* big[2];
  if (c.method == OKLS_METHOD_SHAMPOO) {
    Factor ra = h->fa, rb = h->fb;
    ra.root32 = h->sq_a;
    rb.root32 = h->sq_b;
    Factor* f1[2] = {&ra, &rb};
    int nb = chain_factor_list(f1, 2, c.ns_split_iters, big);
    okls_status s = build_chain(h->chain[0], big, nb, h->sched, c.ns_split_iters, h->scal, sld, true, h->sms);
    if (s != OKLS_OK) return s;
    Factor qa = h->fa, qb = h->fb;
    qa.S = h->sq_a;
    qa.S_upper_only = false;
    qb.S = h->sq_b;
    qb.S_upper_only = false;
    Factor* f2[2] = {&qa, &qb};
    nb = chain_factor_list(f2, 2, c.ns_split_iters, big);
    return build_chain(h->chain[1], big, nb, h->sched, c.ns_split_iters, h->scal, sld, false, h->sms);
  }
  Factor* fs[2] = {&h->fa, &h->fb};
  const int nb = chain_factor_list(fs, 2, c.ns_split_iters, big);
  return build_chain(h->chain[0], big, nb, h->sched, c.ns_split_iters, h->scal, sld, false, h->sms);
}

}  // namespace

// ================================================================== C entries
extern "C" {

int32_t okls_abi_version(void) { return OKLS_ABI_VERSION; }

const char* okls_last_error(void) { return g_err.c_str(); }

okls_status okls_config_default(okls_config* cfg, int64_t batch, int64_t m, int64_t n) {
  if (!cfg) return fail(OKLS_ERR_INVALID_ARG, "config is NULL");
  memset(cfg, 0, sizeof(*cfg));
  cfg->batch = batch;
  cfg->m = m;
  cfg->n = n;
  cfg->param_dtype = OKLS_F32;
  cfg->grad_dtype = OKLS_F32;
  cfg->lr_peak = 0.09434f;
  cfg->beta1 = 0.9684f;
  cfg->beta2 = 0.9482f;
  cfg->eps = 1e-9f;
  cfg->weight_decay = 0.0303f;
  cfg->ns_iters = 10;
  cfg->ns_split_iters = 0;
  cfg->ns_lo = 1e-3f;
  cfg->ridge = 1e-3f;
  cfg->variance_correction = 1;
  cfg->eps_every_update = 1;
  cfg->root_every = 1;
  return OKLS_OK;
}

okls_status okls_state_bytes(const okls_config* cfg, size_t* state_bytes, size_t* workspace_bytes) {
  okls_status s = validate(cfg);
  if (s != OKLS_OK) return s;
  Layout lay;
  s = plan(*cfg, nullptr, nullptr, nullptr, &lay);
  if (s != OKLS_OK) return s;
  if (state_bytes) *state_bytes = lay.state_bytes;
  if (workspace_bytes) *workspace_bytes = lay.ws_bytes;
  return OKLS_OK;
}

okls_status okls_create(const okls_config* cfg, void* state_dev, size_t state_bytes, void* workspace_dev,
                        size_t workspace_bytes, okls_handle* out) {
  if (!out) return fail(OKLS_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  okls_status s = validate(cfg);
  if (s != OKLS_OK) return s;
  if (!state_dev || !workspace_dev) return fail(OKLS_ERR_INVALID_ARG, "state/workspace pointer is NULL");
  if (!aligned(state_dev, 256) || !aligned(workspace_dev, 256))
    return fail(OKLS_ERR_UNSUPPORTED, "state and workspace must be 256-byte aligned");
  Layout lay;
  s = plan(*cfg, nullptr, nullptr, nullptr, &lay);
  if (s != OKLS_OK) return s;
  if (state_bytes < lay.state_bytes || workspace_bytes < lay.ws_bytes)
    return fail(OKLS_ERR_INVALID_ARG, "state needs %zu bytes, workspace %zu bytes", lay.state_bytes, lay.ws_bytes);
  int sms = 0;
  if ((s = device_sms(&sms)) != OKLS_OK) return s;
  okls_handle_s* h = new okls_handle_s();
  h->cfg = *cfg;
  h->sms = sms;
  h->sched = make_schedule(cfg->ns_iters, cfg->ns_lo);
  s = plan(*cfg, static_cast<uint8_t*>(state_dev), static_cast<uint8_t*>(workspace_dev), h, &lay);
  if (s == OKLS_OK && h->nchain > 0) s = build_chains(h);
  if (s != OKLS_OK) {
    delete h;
    return s;
  }
  *out = h;
  return OKLS_OK;
}

okls_status okls_reset_state(okls_handle h, void* stream) {
  if (!h) return fail(OKLS_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const okls_config& c = h->cfg;
  if (c.method == OKLS_METHOD_CLEAN) {
    OKLS_CK(cudaMemsetAsync(h->status, 0, 4, st));
    OKLS_CK(launch_clean_reset(clean_args(h), st));
    h->t = 0;
    return OKLS_OK;
  }
  if (c.method == OKLS_METHOD_SOAP) {
    OKLS_CK(cudaMemsetAsync(h->status, 0, 4, st));
    OKLS_CK(launch_soap_reset(h->M, h->V, h->Sa, h->Sb, h->Pa, h->Pb, static_cast<int>(c.batch), static_cast<int>(c.m),
                              static_cast<int>(c.n), st));
    h->t = 0;
    return OKLS_OK;
  }
  OKLS_CK(cudaMemsetAsync(h->M, 0, static_cast<size_t>(c.batch * c.m * c.n * 4), st));
  OKLS_CK(cudaMemsetAsync(h->scal, 0, static_cast<size_t>(SC_COUNT * c.batch * 4), st));
  OKLS_CK(cudaMemsetAsync(h->status, 0, 4, st));
  OKLS_CK(launch_reset_factor(h->Sa, h->Pa, h->fa.Ph[0].p, nullptr, h->fa.Ph[1].p, nullptr,
                              static_cast<int>(c.m), h->fa.Ph[0].ld, h->fa.Ph[0].mat(), static_cast<int>(c.batch),
                              c.eps, h->scal,
                              static_cast<int>(c.batch), SC_PI_A, st));
  OKLS_CK(launch_reset_factor(h->Sb, h->Pb, h->fb.Ph[0].p, nullptr, h->fb.Ph[1].p, nullptr,
                              static_cast<int>(c.n), h->fb.Ph[0].ld, h->fb.Ph[0].mat(), static_cast<int>(c.batch),
                              c.eps, h->scal,
                              static_cast<int>(c.batch), SC_PI_B, st));
  h->t = 0;
  return OKLS_OK;
}

okls_status okls_step(okls_handle h, void* W, const void* G, float lr, void* stream) {
  return step_impl(h, W, G, lr, nullptr, stream);
}

okls_status okls_step_noise(okls_handle h, void* W, const void* G, float lr, const float* noise, void* stream) {
  return step_impl(h, W, G, lr, noise, stream);
}

}  // extern "C"

namespace {

okls_status step_impl(okls_handle h, void* W, const void* G, float lr, const float* noise, void* stream) {
  if (!h) return fail(OKLS_ERR_INVALID_ARG, "handle is NULL");
  if (!W || !G) return fail(OKLS_ERR_INVALID_ARG, "W or G is NULL");
  if (!aligned(W, 16) || !aligned(G, 16)) return fail(OKLS_ERR_UNSUPPORTED, "W and G must be 16-byte aligned");
  if (!finite_nonneg(lr)) return fail(OKLS_ERR_INVALID_ARG, "lr must be finite and >= 0");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const okls_config& c = h->cfg;
  if (c.method == OKLS_METHOD_CLEAN) return clean_step(h, W, G, lr, noise, st);
  if (c.method == OKLS_METHOD_SOAP) return soap_step(h, W, G, lr, st);
  const bool shampoo = c.method == OKLS_METHOD_SHAMPOO;
  const int B = static_cast<int>(c.batch), m = static_cast<int>(c.m), n = static_cast<int>(c.n);
  const int sld = B;
  const int64_t t1 = h->t + 1;
  // Shampoo: no momentum, N = G
  const float b1 = shampoo ? 0.0f : c.beta1;
  const float kappa = (!shampoo && c.variance_correction) ? static_cast<float>(variance_kappa(c.beta1, t1)) : 1.0f;
  float* M = shampoo ? nullptr : h->M;
  const int gbf = c.grad_dtype == OKLS_BF16;
  const int h12 = kHeadroom;
  const int K = h->sched.iters;
  const int zK = h->sched.z[K], zK1 = h->sched.z[K - 1];
  okls_status s;
  ProfScope scope(&h->prof);
  BoxScope boxes(&h->boxes);
  WaitScope waits(h->wait);

  // 1-2. momentum, statistics, packed binary16 operands
  OKLS_CK(cudaMemsetAsync(h->scal, 0, static_cast<size_t>(4 * B * 4), st));  // SC_SUMSQ_* slots
  const double elems = static_cast<double>(B) * m * n;
  const double gsz = gbf ? 2.0 : 4.0;
  if ((s = bw_launch(elems * (gsz + (M ? 4.0 : 0.0)), st, [&] {
         return launch_momentum_stats(G, gbf, M, B, static_cast<int64_t>(m) * n, b1, kappa, h->part_g, h->part_g_ld,
                                      h->status, st);
       })) != OKLS_OK)
    return s;
  OKLS_CK(launch_coeffs_pre(B, m, n, c.beta2, shampoo ? 1 : 0, h->scal, sld, h->part_g, h->part_g_ld, st));
  note_kernels(1);
  // row pitches: Ghat and Nhat are m x n (pitch ldn), Ghat^T is n x m (pitch ldm)
  if (h->Gh.ld < n || h->GhT.ld < m || h->Gh.rows != m || h->GhT.rows != n ||
      (!shampoo && h->Nh.ld != h->Gh.ld))
    return fail(OKLS_ERR_UNSUPPORTED, "internal plan error: packed operand pitches");
  // G read; M read and written; Ghat, Ghat^T (and Nhat) written
  if ((s = bw_launch(elems * (gsz + (M ? 8.0 : 0.0) + 4.0 + (shampoo ? 0.0 : 2.0)), st, [&] {
         return launch_pack(G, gbf, M, h->Gh.p, h->GhT.p, shampoo ? nullptr : h->Nh.p, B, m, n,
                            /*ldm=*/h->GhT.ld, /*ldn=*/h->Gh.ld, b1, kappa, h->scal, sld, h->status, st);
       })) != OKLS_OK)
    return s;
  // 3. OKLS: X_b = G P_b and X_a^T = G^T P_a^T (previous roots); Shampoo
  //    feeds G itself to the factor products
  const Buf* Xa = &h->XaT;
  const Buf* Xl = &h->Xb;
  if (shampoo) {
    Xl = &h->Gh;
    Xa = &h->GhT;
  } else {
    LaunchBuilder lb;
    GemmProblem& p0 = lb.add_bsplit(h->Gh, h->fb.Ph, h->fb.split, m, n, n, B, EPI_X16, true);
    set_out16(p0, h->Xb, nullptr, nullptr, nullptr);
    p0.alpha = std::ldexp(1.0f, -h12);
    p0.check_finite = 1;
    GemmProblem& p1 = lb.add_bsplit(h->GhT, h->fa.Ph, h->fa.split, n, m, m, B, EPI_X16);
    set_out16(p1, h->XaT, nullptr, nullptr, nullptr);
    p1.alpha = std::ldexp(1.0f, -h12);
    p1.check_finite = 1;
    if ((s = lb.go(h->maps, h->status, h->sms, st)) != OKLS_OK) return s;
  }
  // 4. factor updates on upper tiles (OKLS: EMA, + eps I; Shampoo: plain
  //    sum), the lower triangle mirrored later, with ||S||_F^2 partials
  {
    const float beta = shampoo ? 1.0f : c.beta2;
    const float eps_u = (!shampoo && c.eps_every_update) ? c.eps : 0.0f;
    LaunchBuilder lb;
    GemmProblem& pa = lb.add(Xl, Xl, false, m, m, n, B, EPI_SYRK, true);
    pa.out32 = h->Sa;
    pa.ld32 = m;
    pa.mat32 = static_cast<int64_t>(m) * m;
    pa.scal = h->scal;
    pa.scal_ld = sld;
    pa.scal_slot = SC_ALPHA_SA;
    pa.part = h->part_a;
    pa.part_ld = h->part_a_ld;
    pa.beta = beta;
    pa.gamma = eps_u;
    GemmProblem& pb = lb.add(Xa, Xa, false, n, n, m, B, EPI_SYRK, true);
    pb.out32 = h->Sb;
    pb.ld32 = n;
    pb.mat32 = static_cast<int64_t>(n) * n;
    pb.scal = h->scal;
    pb.scal_ld = sld;
    pb.scal_slot = SC_ALPHA_SB;
    pb.part = h->part_b;
    pb.part_ld = h->part_b_ld;
    pb.beta = beta;
    pb.gamma = eps_u;
    if ((s = lb.go(h->maps, h->status, h->sms, st)) != OKLS_OK) return s;
  }
  // 5-6. fresh roots of both factors (every root_every-th step; the steps in
  // between keep P, its binary16 copy and its scales).  The scales pi of the
  // new roots are committed only after the chain has run.
  const int64_t every = c.root_every > 1 ? c.root_every : 1;
  const bool fresh = ((t1 - 1) % every) == 0;
  if (fresh) {
    OKLS_CK(launch_coeffs_post(B, c.ridge, zK, zK1, h->scal, sld, kPostRoots, h->status, h->part_a, h->part_a_ld,
                               syrk_parts(m), h->part_b, h->part_b_ld, syrk_parts(n), st));
    note_kernels(1);
    if (shampoo) {
      // L^-1/4 = (L^1/2)^-1/2: the first chain (ridge on L) forms only the
      // square roots, the second (no ridge) their inverse square roots
      Factor ra = h->fa, rb = h->fb;
      ra.root32 = h->sq_a;
      rb.root32 = h->sq_b;
      Factor* f1[2] = {&ra, &rb};
      if ((s = run_ns(f1, 2, h->sched, c.ns_split_iters, c.ridge, h->scal, sld, h->maps, h->status, h->sms, st,
                      nullptr, /*root_only=*/true, h->nchain > 0 ? &h->chain[0] : nullptr)) != OKLS_OK)
        return s;
      if ((s = bw_launch(4.0 * B * static_cast<double>(m) * m, st, [&] {
             return launch_sumsq(h->sq_a, B, static_cast<int64_t>(m) * m, h->part_a, h->part_a_ld, st);
           })) != OKLS_OK)
        return s;
      if ((s = bw_launch(4.0 * B * static_cast<double>(n) * n, st, [&] {
             return launch_sumsq(h->sq_b, B, static_cast<int64_t>(n) * n, h->part_b, h->part_b_ld, st);
           })) != OKLS_OK)
        return s;
      OKLS_CK(launch_coeffs_post(B, 0.0f, zK, zK1, h->scal, sld, kPostRoots, h->status, h->part_a, h->part_a_ld,
                                 sumsq_parts(static_cast<int64_t>(m) * m), h->part_b, h->part_b_ld,
                                 sumsq_parts(static_cast<int64_t>(n) * n), st));
      note_kernels(1);
      Factor qa = h->fa, qb = h->fb;
      qa.S = h->sq_a;
      qa.S_upper_only = false;
      qb.S = h->sq_b;
      qb.S_upper_only = false;
      Factor* f2[2] = {&qa, &qb};
      if ((s = run_ns(f2, 2, h->sched, c.ns_split_iters, 0.0f, h->scal, sld, h->maps, h->status, h->sms, st,
                      nullptr, false, h->nchain > 1 ? &h->chain[1] : nullptr)) != OKLS_OK)
        return s;
    } else {
      Factor* fs[2] = {&h->fa, &h->fb};
      if ((s = run_ns(fs, 2, h->sched, c.ns_split_iters, c.ridge, h->scal, sld, h->maps, h->status, h->sms, st,
                      nullptr, false, h->nchain > 0 ? &h->chain[0] : nullptr)) != OKLS_OK)
        return s;
    }
    OKLS_CK(launch_coeffs_post(B, c.ridge, zK, zK1, h->scal, sld, kPostCommit | kPostUpdate, h->status, nullptr, 0,
                               0, nullptr, 0, 0, st));
    note_kernels(1);
  } else {
    OKLS_CK(launch_coeffs_post(B, c.ridge, zK, zK1, h->scal, sld, kPostUpdate, h->status, nullptr, 0, 0, nullptr, 0,
                               0, st));
    note_kernels(1);
    // keep the state symmetric: write the lower triangles of the new factors
    for (Factor* f : {&h->fa, &h->fb}) {
      NormaliseArgs A;
      memset(&A, 0, sizeof(A));
      A.S = f->S;
      A.upper_only = 1;
      A.mirror_only = 1;
      A.d = f->d;
      A.scal = h->scal;
      A.scal_ld = sld;
      A.status = h->status;
      // the upper triangle of S read, the lower one written
      if ((s = bw_launch(4.0 * f->batch * static_cast<double>(f->d) * f->d, st,
                         [&] { return launch_normalise(A, f->batch, st); })) != OKLS_OK)
        return s;
    }
  }
  // 7. Q = P_a N (N = G for Shampoo) into the X_b buffer
  {
    LaunchBuilder lb;
    GemmProblem& p = lb.add_asplit(h->fa.Ph, shampoo ? h->Gh : h->Nh, h->fa.split, m, n, m, B, EPI_X16, true);
    set_out16(p, h->Xb, nullptr, nullptr, nullptr);
    p.alpha = std::ldexp(1.0f, -h12);
    p.check_finite = 1;
    if ((s = lb.go(h->maps, h->status, h->sms, st)) != OKLS_OK) return s;
  }
  // 8. U = Q P_b, W <- W (1 - lr wd lr/lr_peak) - lr c_shape U (c_shape = 1 for Shampoo)
  {
    LaunchBuilder lb;
    GemmProblem& p = lb.add_bsplit(h->Xb, h->fb.Ph, h->fb.split, m, n, n, B, EPI_UPDATE, true);
    p.w = W;
    p.w_bf16 = c.param_dtype == OKLS_BF16;
    p.ld32 = n;
    p.mat32 = static_cast<int64_t>(m) * n;
    p.scal = h->scal;
    p.scal_ld = sld;
    p.scal_slot = SC_UCOEF;
    const double cshape =
        shampoo ? 1.0
                : std::sqrt(static_cast<double>(m) / n) / (std::sqrt(static_cast<double>(m)) + std::sqrt(static_cast<double>(n)));
    p.alpha = static_cast<float>(1.0 - static_cast<double>(lr) * c.weight_decay * (static_cast<double>(lr) / c.lr_peak));
    p.beta = static_cast<float>(static_cast<double>(lr) * cshape);
    if ((s = lb.go(h->maps, h->status, h->sms, st)) != OKLS_OK) return s;
  }
  h->t = t1;
  return OKLS_OK;
}

}  // namespace

extern "C" {

okls_status okls_query_status(okls_handle h, void* stream, uint32_t* dev_status) {
  if (!h) return fail(OKLS_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  OKLS_CK(cudaStreamSynchronize(st));
  OKLS_CK(cudaMemcpy(&v, h->status, 4, cudaMemcpyDeviceToHost));
  OKLS_CK(cudaMemset(h->status, 0, 4));
  if (dev_status) *dev_status = v;
  if (v & kStTimeout) return fail(OKLS_ERR_TIMEOUT, "a device-side wait expired (status 0x%x)", v);
  if (v) return fail(OKLS_ERR_NONFINITE, "non-finite values in the step (status 0x%x)", v);
  return OKLS_OK;
}

static okls_status part_ptr(okls_handle h, int32_t part, float** p, size_t* bytes) {
  const okls_config& c = h->cfg;
  if (c.method == OKLS_METHOD_CLEAN) {
    const int64_t B = c.batch, m = c.m, n = c.n, r = c.rank;
    int64_t elems = 0;
    switch (part) {
      case OKLS_STATE_M: *p = h->M; elems = B * r * r; break;
      case OKLS_STATE_V: *p = h->V; elems = B * r * r; break;
      case OKLS_STATE_PA: *p = h->Pa; elems = B * m * r; break;
      case OKLS_STATE_PB: *p = h->Pb; elems = B * n * r; break;
      case OKLS_STATE_SA: *p = h->Sa; elems = B * r; break;
      case OKLS_STATE_SB: *p = h->Sb; elems = B * r; break;
      case OKLS_STATE_MA: *p = h->MA; elems = B * m * r; break;
      case OKLS_STATE_MB: *p = h->MB; elems = B * r * n; break;
      case OKLS_STATE_VA: *p = h->vA; elems = B * r; break;
      case OKLS_STATE_VB: *p = h->vB; elems = B * r; break;
      case OKLS_STATE_VC: *p = h->vC; elems = B; break;
      default: return fail(OKLS_ERR_INVALID_ARG, "unknown state part %d", part);
    }
    *bytes = static_cast<size_t>(elems * 4);
    return OKLS_OK;
  }
  switch (part) {
    case OKLS_STATE_M: *p = h->M; *bytes = static_cast<size_t>(c.batch * c.m * c.n * 4); break;
    case OKLS_STATE_SA: *p = h->Sa; *bytes = static_cast<size_t>(c.batch * c.m * c.m * 4); break;
    case OKLS_STATE_SB: *p = h->Sb; *bytes = static_cast<size_t>(c.batch * c.n * c.n * 4); break;
    case OKLS_STATE_PA: *p = h->Pa; *bytes = static_cast<size_t>(c.batch * c.m * c.m * 4); break;
    case OKLS_STATE_PB: *p = h->Pb; *bytes = static_cast<size_t>(c.batch * c.n * c.n * 4); break;
    case OKLS_STATE_V:
      if (c.method != OKLS_METHOD_SOAP)
        return fail(OKLS_ERR_INVALID_ARG, "state part V exists in SOAP and Clean modes only");
      *p = h->V;
      *bytes = static_cast<size_t>(c.batch * c.m * c.n * 4);
      break;
    default: return fail(OKLS_ERR_INVALID_ARG, "unknown state part %d", part);
  }
  return OKLS_OK;
}

okls_status okls_get_state(okls_handle h, int32_t part, void* dst, void* stream) {
  if (!h || !dst) return fail(OKLS_ERR_INVALID_ARG, "handle or dst is NULL");
  float* p = nullptr;
  size_t bytes = 0;
  okls_status s = part_ptr(h, part, &p, &bytes);
  if (s != OKLS_OK) return s;
  OKLS_CK(cudaMemcpyAsync(dst, p, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
  return OKLS_OK;
}

okls_status okls_set_state(okls_handle h, int32_t part, const void* src, void* stream) {
  if (!h || !src) return fail(OKLS_ERR_INVALID_ARG, "handle or src is NULL");
  float* p = nullptr;
  size_t bytes = 0;
  okls_status s = part_ptr(h, part, &p, &bytes);
  if (s != OKLS_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  OKLS_CK(cudaMemcpyAsync(p, src, bytes, cudaMemcpyDeviceToDevice, st));
  const okls_config& c = h->cfg;
  // SOAP's and Clean's bases have no binary16 copies
  if (c.method == OKLS_METHOD_SOAP || c.method == OKLS_METHOD_CLEAN) return OKLS_OK;
  if (part == OKLS_STATE_PA)
    OKLS_CK(launch_requant(h->Pa, static_cast<int>(c.batch), static_cast<int>(c.m), h->fa.Ph[0].p, nullptr,
                           h->fa.Ph[1].p, nullptr, h->fa.Ph[0].ld, h->fa.Ph[0].mat(), h->scal,
                           static_cast<int>(c.batch), SC_PI_A, st));
  if (part == OKLS_STATE_PB)
    OKLS_CK(launch_requant(h->Pb, static_cast<int>(c.batch), static_cast<int>(c.n), h->fb.Ph[0].p, nullptr,
                           h->fb.Ph[1].p, nullptr, h->fb.Ph[0].ld, h->fb.Ph[0].mat(), h->scal,
                           static_cast<int>(c.batch), SC_PI_B, st));
  return OKLS_OK;
}

okls_status okls_get_step(okls_handle h, int64_t* t) {
  if (!h || !t) return fail(OKLS_ERR_INVALID_ARG, "handle or t is NULL");
  *t = h->t;
  return OKLS_OK;
}

okls_status okls_set_step(okls_handle h, int64_t t) {
  if (!h || t < 0) return fail(OKLS_ERR_INVALID_ARG, "bad handle or step");
  h->t = t;
  return OKLS_OK;
}

okls_status okls_destroy(okls_handle h) {
  delete h;
  return OKLS_OK;
}

okls_status okls_set_wait_limit(okls_handle h, int64_t cycles, int64_t unloaded_tile) {
  if (!h) return fail(OKLS_ERR_INVALID_ARG, "handle is NULL");
  if (cycles < 0 || unloaded_tile < -1) return fail(OKLS_ERR_INVALID_ARG, "cycles >= 0, unloaded_tile >= -1");
  h->wait.cycles = cycles;
  h->wait.unloaded_tile = unloaded_tile;
  return OKLS_OK;
}

okls_status okls_profile_enable(okls_handle h, int32_t timing) {
  if (!h) return fail(OKLS_ERR_INVALID_ARG, "handle is NULL");
  h->prof.timing = timing != 0;
  return OKLS_OK;
}

okls_status okls_profile_read(okls_handle h, okls_profile* out) {
  if (!h || !out) return fail(OKLS_ERR_INVALID_ARG, "handle or out is NULL");
  Prof& p = h->prof;
  memset(out, 0, sizeof(*out));
  out->kernel_launches = p.kernels;
  out->gemm_launches = p.gemm_launches;
  out->gemm_flops = p.gemm_flops;
  out->ns_launches = p.ns_launches;
  out->ns_flops = p.ns_flops;
  out->bw_launches = p.bw_launches;
  out->bw_bytes = p.bw_bytes;
  for (const Prof::Rec& r : p.recs) {
    OKLS_CK(cudaEventSynchronize(r.b));
    float ms = 0.0f;
    OKLS_CK(cudaEventElapsedTime(&ms, r.a, r.b));
    if (r.bw) {
      out->bw_ms += ms;
      out->bw_timed_launches += 1;
      continue;
    }
    out->gemm_ms += ms;
    if (r.ns) out->ns_ms += ms;
    out->timed_launches += 1;
  }
  p.recs.clear();
  p.used = 0;
  p.kernels = p.gemm_launches = p.ns_launches = p.bw_launches = 0;
  p.gemm_flops = p.ns_flops = p.bw_bytes = 0.0;
  return OKLS_OK;
}

okls_status okls_ns_schedule(int32_t iters, double lo, double* a, double* b, int32_t* zexp) {
  if (iters < 1 || iters > 64 || !(lo > 0.0 && lo <= 1.0))
    return fail(OKLS_ERR_INVALID_ARG, "iters in [1, 64], lo in (0, 1]");
  Sched s = make_schedule(iters, lo);
  for (int k = 0; k < iters; ++k) {
    if (a) a[k] = s.a[k];
    if (b) b[k] = s.b[k];
  }
  if (zexp)
    for (int k = 0; k <= iters; ++k) zexp[k] = s.z[k];
  return OKLS_OK;
}

// ------------------------------------------------------------ inverse roots
static okls_status inv_plan(int64_t d, int64_t count, int32_t split, uint8_t* ws, Factor* f, float** scal,
                            uint32_t** status, CUtensorMap** maps, size_t* bytes, std::vector<CUtensorMap>* mv,
                            float** part, std::vector<int>* boxes = nullptr) {
  Planner wp;
  wp.base = ws;
  *maps = static_cast<CUtensorMap*>(wp.take(kMapTableBytes, 128));
  *scal = static_cast<float*>(wp.take(static_cast<size_t>(SC_COUNT * count * 4)));
  *status = static_cast<uint32_t*>(wp.take(256));
  *part = static_cast<float*>(wp.take(static_cast<size_t>(count * factor_parts(d) * 4)));
  plan_factor(wp, *f, static_cast<int>(d), static_cast<int>(count), split > 0);
  if (wp.err != OKLS_OK) return wp.err;
  *bytes = wp.off;
  if (mv) *mv = wp.maps;
  if (boxes) *boxes = wp.boxes;
  return OKLS_OK;
}

okls_status okls_inv_root_workspace_bytes(int64_t d, int64_t count, int32_t iters, int32_t split_iters,
                                          size_t* workspace_bytes) {
  if (d < 1 || d > 32768 || count < 1 || count > 65535 || iters < 2 || iters > 32 || split_iters < 0 ||
      split_iters > iters || !workspace_bytes)
    return fail(OKLS_ERR_INVALID_ARG, "bad inverse-root arguments");
  Factor f;
  float* scal;
  uint32_t* status;
  CUtensorMap* maps;
  float* part;
  return inv_plan(d, count, split_iters, nullptr, &f, &scal, &status, &maps, workspace_bytes, nullptr, &part);
}

okls_status okls_inv_root(const float* S, float* P, float* root, uint16_t* trace, int64_t d, int64_t count,
                          int32_t iters, int32_t split_iters, float lo, float ridge, void* ws, size_t ws_bytes,
                          void* stream) {
  size_t need = 0;
  okls_status s = okls_inv_root_workspace_bytes(d, count, iters, split_iters, &need);
  if (s != OKLS_OK) return s;
  if (!S || !P || !ws) return fail(OKLS_ERR_INVALID_ARG, "S, P and workspace must be non-NULL");
  if (ws_bytes < need) return fail(OKLS_ERR_INVALID_ARG, "workspace needs %zu bytes", need);
  if (!aligned(ws, 256)) return fail(OKLS_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
  if (!(lo > 0.0f && lo < 1.0f) || !finite_nonneg(ridge)) return fail(OKLS_ERR_INVALID_ARG, "bad lo or ridge");
  int sms = 0;
  if ((s = device_sms(&sms)) != OKLS_OK) return s;
  Factor f;
  float* scal;
  uint32_t* status;
  CUtensorMap* maps;
  float* part;
  std::vector<CUtensorMap> mv;
  std::vector<int> box_rows;
  if ((s = inv_plan(d, count, split_iters, static_cast<uint8_t*>(ws), &f, &scal, &status, &maps, &need, &mv,
                    &part, &box_rows)) != OKLS_OK)
    return s;
  BoxScope boxes(&box_rows);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  OKLS_CK(cudaMemcpyAsync(maps, mv.data(), mv.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice, st));
  OKLS_CK(cudaMemsetAsync(scal, 0, static_cast<size_t>(SC_COUNT * count * 4), st));
  OKLS_CK(cudaMemsetAsync(status, 0, 4, st));
  f.S = const_cast<float*>(S);
  f.P32 = P;
  f.root32 = root;
  f.slot_sumsq = SC_SUMSQ_SA;
  f.slot_cprime = SC_CPRIME_A;
  f.slot_pi = SC_PI_A;
  f.slot_pscale = SC_PSCALE_A;
  f.slot_rscale = SC_RSCALE_A;
  const Sched sc = make_schedule(iters, lo);
  OKLS_CK(launch_sumsq(S, static_cast<int>(count), d * d, part, factor_parts(d), st));
  OKLS_CK(launch_coeffs_post(static_cast<int>(count), ridge, sc.z[iters], sc.z[iters - 1], scal,
                             static_cast<int>(count), kPostRoots, status, part, factor_parts(d), sumsq_parts(d * d),
                             nullptr, 0, 0, st));
  TraceOut tr;
  tr.base = trace;
  tr.count = count;
  tr.d = d;
  Factor* fs[1] = {&f};
  s = run_ns(fs, 1, sc, split_iters, ridge, scal, static_cast<int>(count), maps, status, sms, st, &tr);
  // keep the host descriptor table alive until the upload has run
  cudaError_t e = cudaStreamSynchronize(st);
  if (s != OKLS_OK) return s;
  if (e != cudaSuccess) return fail(OKLS_ERR_CUDA, "inverse root: %s", cudaGetErrorString(e));
  uint32_t v = 0;
  OKLS_CK(cudaMemcpy(&v, status, 4, cudaMemcpyDeviceToHost));
  if (v & kStTimeout) return fail(OKLS_ERR_TIMEOUT, "a device-side wait expired (status 0x%x)", v);
  if (v) return fail(OKLS_ERR_NONFINITE, "non-finite Newton-Schulz iterate (status 0x%x)", v);
  return OKLS_OK;
}

}  // extern "C"

// ===================================================== no-allocation variant
// Some callers cannot allocate device memory at the moment they need an
// inverse root: allocators that must not re-enter themselves and embedders
// whose memory pool is fixed at start-up.  For them okls_inv_root_noalloc
// takes its scratch from this file-scope array instead of a caller-provided
// workspace.  Every GPU that loads the library holds it (32 MiB) until the
// process exits.  The call is not usable under stream capture: it uploads a
// host-side descriptor table and synchronises the stream.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the array's name in host code is only a host-side stand-in).
okls_status noalloc_scratch(void** out) {
  int dev = 0;
  OKLS_CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(OKLS_ERR_NO_DEVICE, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(OKLS_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return OKLS_OK;
}

}  // namespace

extern "C" {

size_t okls_inv_root_noalloc_capacity(void) { return kNoAllocScratchBytes; }

okls_status okls_inv_root_noalloc(const float* S, float* P, int64_t d, int64_t count, int32_t iters,
                                  int32_t split_iters, float lo, float ridge, void* stream) {
  size_t need = 0;
  okls_status s = okls_inv_root_workspace_bytes(d, count, iters, split_iters, &need);
  if (s != OKLS_OK) return s;
  if (need > kNoAllocScratchBytes)
    return fail(OKLS_ERR_UNSUPPORTED,
                "okls_inv_root_noalloc: %lld matrices of %lld x %lld need %zu bytes of scratch; the static "
                "scratch holds %zu bytes (use okls_inv_root with a workspace)",
                static_cast<long long>(count), static_cast<long long>(d), static_cast<long long>(d), need,
                kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != OKLS_OK) return s;
  // the shared scratch keeps the previous call's contents; okls_inv_root
  // clears the scalar sums and the status word it relies on
  s = okls_inv_root(S, P, nullptr, nullptr, d, count, iters, split_iters, lo, ridge, scratch, kNoAllocScratchBytes,
                    stream);
  // some error paths of okls_inv_root return before its final
  // synchronisation: drain the stream so that no work of this call is still
  // queued on the shared array when the next call starts (the error message
  // of the failed call is kept)
  if (s != OKLS_OK) (void)cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  return s;
}

}  // extern "C"

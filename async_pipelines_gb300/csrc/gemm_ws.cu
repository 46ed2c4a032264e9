// Host side of the C ABI declared in include/gemm_ws.h: argument checks (the
// `can_implement` role of "sm90_gemm_tma_warpspecialized_cooperative.hpp"),
// TMA descriptor encoding (cached per handle), the device workspace (counters,
// status word, stream-K partials), the per-problem plan (tile configuration,
// half-width tail units, quarter-width units for tiny problems or stream-K
// pieces, persistent grid of at most the co-resident clusters) and the
// launches: the GEMM, one CTA per SM, and after split tiles the reduction of
// their pieces.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_ws.h"
#ifdef GEMM_WS_DEBUG
#include "gemm_ws_debug.h"
#endif
#include "gemm_ws_kernel.cuh"

// A tensor map the handle encoded before, and what it describes.
struct MapCacheEntry {
  const void* ptr;
  uint64_t d0, d1, d2;
  uint32_t b0, b1;
  int swizzle, promotion;
  bool valid;
  CUtensorMap map;
};
constexpr int kMapCache = 16;

struct gemm_ws {
  int device;
  int num_sms;
  int cta_group;                  // 0: chosen per problem (default); 1: single-CTA tiles; 2: CTA pairs
  int pdl;                        // launch with programmatic stream serialisation
  int group_m;                    // raster group: m-tiles walked per n step
  int max_pair_clusters;          // co-resident 2-CTA clusters of the pair kernel
  int stream_k;                   // 0 off, 1 where the cost model gains (default), 2 always
  int sk_inline;                  // two-piece tiles: fix-up inside the GEMM (default 1)
  int k_snake;                    // every other unit of a cluster walks K backwards
  uint32_t* work;                 // [0] stream-out counter, [1] status, [2] done count, then
                                  // the in-kernel fix-up words (work_words)
  float* partial;                 // stream-K partials: num_sms parts of 128 x 256 fp32
  int last_cuda_error;
  unsigned long long timeout_ns;
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  MapCacheEntry map_cache[kMapCache];   // recently encoded tensor maps (host memory)
  int map_cache_next;
#ifdef GEMM_WS_DEBUG
  int debug_fault;
  unsigned long long* trace;
  unsigned long long* phases;
#endif
};

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int64_t kMaxElems = int64_t{1} << 40;
constexpr int kWorkWords = 4;   // counter [0], status [1], consumers done [2]

// Words of a handle's work area: kWorkWords, then the in-kernel fix-up's
// arrival counts and written flags (one per epilogue warp of each CTA).
size_t work_words(int num_sms) {
  return kWorkWords + 2 * static_cast<size_t>(num_sms) * gws::NUM_EPI_WARPS;
}

int cuda_fail(gemm_ws* h, cudaError_t e) {
  if (h) h->last_cuda_error = static_cast<int>(e);
  return GEMM_WS_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// A 3-D bf16 tensor {d0 (contiguous), d1, d2}, packed, tiled box {b0, b1, 1}.
// Encodings are cached per handle (the map depends only on these values), so
// repeated calls on the same buffers skip the driver's encoder.
CUresult encode3d(gemm_ws* h, CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw,
                  CUtensorMapL2promotion promo) {
  for (int i = 0; i < kMapCache; ++i) {
    const MapCacheEntry& e = h->map_cache[i];
    if (e.valid && e.ptr == ptr && e.d0 == d0 && e.d1 == d1 && e.d2 == d2 && e.b0 == b0 &&
        e.b1 == b1 && e.swizzle == static_cast<int>(sw) &&
        e.promotion == static_cast<int>(promo)) {
      std::memcpy(m, &e.map, sizeof(CUtensorMap));
      return CUDA_SUCCESS;
    }
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      h->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    MapCacheEntry& e = h->map_cache[h->map_cache_next];
    h->map_cache_next = (h->map_cache_next + 1) % kMapCache;
    e.ptr = ptr;
    e.d0 = d0;
    e.d1 = d1;
    e.d2 = d2;
    e.b0 = b0;
    e.b1 = b1;
    e.swizzle = static_cast<int>(sw);
    e.promotion = static_cast<int>(promo);
    e.map = *m;
    e.valid = true;
  }
  return r;
}

int check_problem(gemm_ws* h, const uint16_t* A, const uint16_t* B, const uint16_t* C,
                  uint16_t* D, int64_t M, int64_t N, int64_t K, int64_t L, float beta) {
  if (!h) return GEMM_WS_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || L < 0) return GEMM_WS_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim || L > kMaxDim) return GEMM_WS_ERR_INVALID_ARG;
  if (M * N * L == 0) return GEMM_WS_OK;   // nothing to do; pointers unchecked
  if (L * M > kMaxElems / (N > 0 ? N : 1) || L * M > kMaxElems / (K > 0 ? K : 1) ||
      L * N > kMaxElems / (K > 0 ? K : 1))
    return GEMM_WS_ERR_INVALID_ARG;
  if (!D) return GEMM_WS_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B)) return GEMM_WS_ERR_INVALID_ARG;
  if (beta != 0.0f && !C) return GEMM_WS_ERR_INVALID_ARG;
  if ((K % 8) != 0 || (N % 8) != 0) return GEMM_WS_ERR_ALIGNMENT;
  if (!aligned16(D) || (K > 0 && (!aligned16(A) || !aligned16(B))) ||
      (beta != 0.0f && !aligned16(C)))
    return GEMM_WS_ERR_ALIGNMENT;
  const int64_t dbytes = 2 * L * M * N;
  if (K > 0 && (overlaps(D, dbytes, A, 2 * L * M * K) || overlaps(D, dbytes, B, 2 * L * N * K)))
    return GEMM_WS_ERR_INVALID_ARG;
  if (beta != 0.0f && C != D && overlaps(D, dbytes, C, dbytes)) return GEMM_WS_ERR_INVALID_ARG;
  return GEMM_WS_OK;
}

// How many of the last tiles (in raster order) to run as two half-width
// units so that the persistent schedule's final wave is not half idle.
// Cluster c runs units c, c + P, ...; a whole tile costs 1, a half ~0.8
// (same k-loop and A traffic, half the MMA work: load-bound; 0.79 measured on
// GB300 at 4096^3). Returns the number of whole tiles (and, in *cost, the
// slowest cluster's work in tile units); only
// splits of at most one wave of tiles are considered (with fewer tiles than
// clusters, splitting spreads a small problem over more SMs).
int64_t choose_num_full(int64_t tiles, int64_t P, double* cost) {
  if (P <= 1) {
    *cost = static_cast<double>(tiles);
    return tiles;
  }
  // Cluster c gets ceil-or-floor shares of both the units and the whole
  // tiles, both non-increasing in c, so cluster 0 is always the slowest.
  double best = 0.0;
  int64_t best_full = tiles;
  for (int64_t s = 0; s <= P && s <= tiles; ++s) {
    const int64_t F = tiles - s, U = F + 2 * s;
    const int64_t n_full = (F + P - 1) / P, n_units = (U + P - 1) / P;
    const double worst =
        static_cast<double>(n_full) + 0.8 * static_cast<double>(n_units - n_full);
    if (s == 0 || worst < best - 1e-9) {
      best = worst;
      best_full = F;
    }
  }
  *cost = best;
  return best_full;
}

// Co-resident clusters of `cs` CTAs of kernel `fn` on the current device.
template <typename F>
cudaError_t max_clusters(F fn, int cs, int num_sms, uint32_t smem, int* out) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cs * (num_sms / cs), 1, 1);
  cfg.blockDim = dim3(gws::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, fn, &cfg);
}

// Sets the shared-memory attribute of both kernel instances on the current
// device and returns how many 2-CTA clusters fit at once.
cudaError_t configure_kernels(int num_sms, int* max_pair_clusters) {
  cudaError_t e = cudaFuncSetAttribute(gws::gemm_ws_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(gws::Cfg<1>::SMEM_BYTES));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gws::gemm_ws_kernel<2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(gws::Cfg<2>::SMEM_BYTES));
  if (e == cudaSuccess)
    e = max_clusters(gws::gemm_ws_kernel<2>, 2, num_sms, gws::Cfg<2>::SMEM_BYTES,
                     max_pair_clusters);
  return e;
}

// Wide (32 x 64) D stores for K up to this (see launch).
constexpr int64_t kWideDMaxK = 512;

// Persistent clusters the launch may use: SMs for single CTAs, else the
// co-resident CTA pairs.
int64_t cluster_capacity(const gemm_ws* h, int cs) {
  return cs == 1 ? h->num_sms : h->max_pair_clusters;
}

// Stream-K pieces. The tiles of a stream-K region (the last tiles in raster
// order) have their K ranges cut into S equal pieces, each run by its own
// cluster as that cluster's last unit; pieces with the same index sit at the
// same k on every tile, so concurrent tiles still share A and B panels
// through L2. The pieces are added in piece order, and the alpha/beta
// epilogue of those tiles runs after the sum:
//  - two pieces (sk_inline): inside the GEMM. Per epilogue warp, the piece
//    that arrives second takes the other's fp32 partial (written to the
//    workspace and flagged) and runs the epilogue; it waits only for a piece
//    that has already arrived, so the GEMM needs no co-resident clusters.
//  - more pieces: every piece writes its partial and waits for nothing; a
//    reduction kernel that follows the GEMM on the stream adds them (the
//    separate-reduction variant of the SM90 cooperative kernel's fix-up).
//    One piece adding all the others' partials would move S - 1 partials
//    through one SM.
//  - Few tiles (at most half as many as clusters): every tile, S =
//    min(clusters / tiles, K / kMinShareK, kMaxSplit) (split-K).
//  - Otherwise the tiles of the last, partial wave if it is at most half
//    full: S = min(clusters / those tiles, ...) and the waves before it run
//    whole tiles (instead of running that wave as half-width tiles, which
//    cost ~0.8 of a whole one on GB300 because they are load-bound).
// The default (GEMM_WS_STREAM_K=1) takes the split where the host cost model
// (tile-times of the slowest cluster; kPieceCostStages of fix-up per piece)
// beats whole tiles with half-width tails; GEMM_WS_STREAM_K=2 takes it
// wherever the shape allows, with pieces down to one ring stage (tests).
constexpr int64_t kMinShareK = 1024;
constexpr int64_t kMaxSplit = 16;
constexpr int64_t kMaxSplitForced = 32;
// Fix-up cost of a split tile, in ring stages of MMA work (~0.5-0.6 us each
// on GB300): the pieces' partial writes, their reduction (in the GEMM for two
// pieces, else by the reduction kernel after it) and a short piece's
// pipeline fill. Calibrated by timing: 10 splits 8192^3's and 1536^2 x
// 8192's tails and leaves 4096^3's and 8192^2 x 4096's (32-stage tiles) to
// half-width tiles. Split with the in-kernel fix-up, interleaved against
// half-width tails: 8192^3 -0.6 %, 4096^3 +2.4 %, 8192^2 x 4096 +1.2 %; with
// the reduction kernel 4096^3 was +4 %.
constexpr double kPieceCostStages = 10.0;
constexpr size_t kPartBytes = size_t{gws::BM} * gws::BN * sizeof(float);
// Workspace: one partial part per CTA of a launch (each runs at most one
// piece).
#ifdef GEMM_WS_DEBUG
constexpr int kScheduleCols = 15;   // columns of a gemm_ws_debug_schedule row
#endif

struct Plan {
  int cg;              // CTA group of the MMA (1 or 2)
  int cs;              // CTAs per cluster
  int64_t tiles_m, tiles_n, num_tiles;
  int64_t num_full;    // whole-width units (the rest of the tiles run as `split` parts)
  int64_t split;       // 2: halves, 4: quarters
  int64_t num_units;   // units (an upper bound of unit ids with stream-K)
  int64_t num_stages;  // ring stages covering K
  int64_t sk_first;    // first tile of the stream-K region (num_tiles: none)
  int64_t sk_split;    // pieces per tile of the region
  int64_t sk_clusters; // clusters running pieces
  bool sk_inline;      // two-piece tiles fixed up inside the GEMM (no reduction kernel)
  int64_t clusters;    // persistent clusters launched
};

// Tile configuration of one problem: single-CTA 128 x 256 tiles where the
// work per tile is short (K <= 512: the epilogue, not the MMA, bounds it) or
// the problem is small (K <= 1024 with at most two waves of pair tiles), CTA
// pairs with 256 x 256 tiles otherwise. Measured on GB300 over M = N in
// 256..8192, K in 64..8192: single CTAs are 16-33 % faster at K <= 256 and
// up to 14 % at K = 1024 on small problems; pairs 7-18 % faster for K >= 2048
// on larger ones. The handle can force either (GEMM_WS_CTA_GROUP).
int pick_cta_group(const gemm_ws* h, int64_t M, int64_t N, int64_t K, int64_t L) {
  if (h->cta_group == 1 || h->max_pair_clusters < 1) return 1;
  if (h->cta_group == 2) return 2;
  const int64_t pair_tiles = L * ((M + 2 * gws::BM - 1) / (2 * gws::BM)) * ((N + gws::BN - 1) / gws::BN);
  if (K <= 512 || (K <= 1024 && pair_tiles <= 2 * static_cast<int64_t>(h->max_pair_clusters)))
    return 1;
  return 2;
}

// The persistent schedule of one launch: host arithmetic only, shared by the
// launch and the debug query.
Plan make_plan(const gemm_ws* h, int64_t M, int64_t N, int64_t K, int64_t L, bool streamout) {
  Plan q;
  const int cg = pick_cta_group(h, M, N, K, L);
  q.cg = cg;
  q.cs = cg;
  q.tiles_m = (M + gws::BM * q.cs - 1) / (gws::BM * q.cs);
  q.tiles_n = (N + gws::BN - 1) / gws::BN;
  q.num_tiles = L * q.tiles_m * q.tiles_n;
  const int64_t ksub = cg == 1 ? gws::Cfg<1>::KSUB : gws::Cfg<2>::KSUB;
  const int64_t T = q.num_tiles;
  const int64_t ns = ((K + gws::BK - 1) / gws::BK + ksub - 1) / ksub;
  q.num_stages = ns;
  const int64_t P = cluster_capacity(h, q.cs);
  double dp_cost = 0.0;
  q.num_full = choose_num_full(T, P, &dp_cost);
  q.split = 2;
  q.num_units = q.num_full + 2 * (T - q.num_full);
  q.clusters = q.num_units < P ? q.num_units : P;
  q.sk_first = T;
  q.sk_split = 1;
  q.sk_clusters = 0;
  q.sk_inline = false;
  // Quarter units for problems of so few tiles that four units per tile fit
  // on the GPU at once (a latency-bound launch: each SM's loads, MMAs and
  // epilogue shrink with the unit), unless split pieces are taken below.
  // Stream-out keeps its 128-column handoff granularity, so no quarters.
  auto quarters = [&](Plan& r) {
    if (!streamout && 4 * T <= P) {
      r.num_full = 0;
      r.split = 4;
      r.num_units = 4 * T;
      r.clusters = r.num_units;
    }
    return r;
  };
  // Stream-out keeps whole tiles: its consumer takes every tile where the
  // epilogue computes it.
  if (streamout || h->stream_k == 0 || !h->partial || P < 2) return quarters(q);
  const bool forced = h->stream_k == 2;
  const int64_t min_share = forced ? 1 : kMinShareK / (gws::BK * ksub);
  const int64_t R = 2 * T <= P ? T : T % P;   // tiles of the stream-K region
  if (R == 0 || 2 * R > P) return quarters(q);
  int64_t S = P / R;
  if (S > ns / min_share) S = ns / min_share;
  if (S > (forced ? kMaxSplitForced : kMaxSplit)) S = forced ? kMaxSplitForced : kMaxSplit;
  if (S < 2) return quarters(q);
  const int64_t F = T - R, Pe = R * S;
  const bool inl = S == 2 && h->sk_inline;
  const double sk_cost = static_cast<double>(F / P) + static_cast<double>((ns + S - 1) / S) / ns +
                         kPieceCostStages / static_cast<double>(ns);
  if (!forced && !(sk_cost < dp_cost - 1e-9)) return quarters(q);
  q.sk_first = F;
  q.sk_split = S;
  q.sk_inline = inl;
  q.sk_clusters = Pe;
  q.num_full = T;
  q.num_units = F + Pe;
  q.clusters = F > 0 ? P : Pe;
  return q;
}

int launch(gemm_ws* h, const uint16_t* A, const uint16_t* B, const uint16_t* C, uint16_t* D,
           int64_t M, int64_t N, int64_t K, int64_t L, float alpha, float beta,
           uint16_t* staging, uint32_t* flags, cudaStream_t stream) {
  gws::Params p;
  std::memset(&p, 0, sizeof p);
  const Plan q = make_plan(h, M, N, K, L, staging != nullptr);
  const int cg = q.cg;
  const int cs = q.cs;   // CTAs per cluster
  if (q.num_units > kMaxDim) return GEMM_WS_ERR_INVALID_ARG;
  const int64_t stn = (N + gws::STAGING - 1) / gws::STAGING;
  const int64_t T = L * ((M + gws::STAGING - 1) / gws::STAGING) * stn;
  if (T > kMaxDim) return GEMM_WS_ERR_INVALID_ARG;

  CUresult r = CUDA_SUCCESS;
  if (K > 0) {
    r = encode3d(h, &p.tmA, A, K, M, L, gws::BK, gws::BM, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r == CUDA_SUCCESS)
      r = encode3d(h, &p.tmB, B, K, N, L, gws::BK, gws::BN / cs, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r == CUDA_SUCCESS && q.num_full < q.num_tiles)
      r = encode3d(h, q.split == 4 ? &p.tmB4 : &p.tmB2, B, K, N, L, gws::BK,
                   static_cast<uint32_t>(gws::BN / q.split / cs), CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  }
  if (r == CUDA_SUCCESS && beta != 0.0f)
    r = encode3d(h, &p.tmC, C, N, M, L, gws::EPI_N, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (r == CUDA_SUCCESS)
    r = encode3d(h, &p.tmD, D, N, M, L, gws::EPI_N, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  // Wide D stores (32 x 64 blocks): measured on GB300 against 32 x 32 blocks,
  // interleaved: 8192^2 x 64 -24 %, 8192^2 x 256 -14 %, 4096^2 x 256 -12 %,
  // 2048^2 x 512 -2 %; 4096^3 +1 %, 8192^2 x 1024 +4 %.
  const bool wide_d = beta == 0.0f && !staging && q.sk_first == q.num_tiles && K <= kWideDMaxK;
  if (r == CUDA_SUCCESS && wide_d)
    r = encode3d(h, &p.tmDw, D, N, M, L, 2 * gws::EPI_N, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (r == CUDA_SUCCESS && staging)
    r = encode3d(h, &p.tmS, staging, gws::STAGING, gws::STAGING, static_cast<uint64_t>(T),
                 gws::EPI_N, gws::STAGING, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (r != CUDA_SUCCESS) {
    h->last_cuda_error = static_cast<int>(r);
    return GEMM_WS_ERR_CUDA;
  }

  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.L = static_cast<int>(L);
  p.tiles_m = static_cast<int>(q.tiles_m);
  p.tiles_n = static_cast<int>(q.tiles_n);
  p.num_tiles = static_cast<int>(q.num_tiles);
  p.num_full = static_cast<int>(q.num_full);
  p.split = static_cast<int>(q.split);
  p.num_units = static_cast<int>(q.num_units);
  p.num_kb = static_cast<int>((K + gws::BK - 1) / gws::BK);
  p.num_stages = static_cast<int>(q.num_stages);
  p.sk_first = static_cast<int>(q.sk_first);
  p.sk_split = static_cast<int>(q.sk_split);
  p.partial = h->partial;
  p.sk_inline = q.sk_inline ? 1 : 0;
  p.sk_sync = q.sk_inline ? h->work + kWorkWords : nullptr;
  p.group_m = h->group_m;
  p.k_snake = h->k_snake;
  p.staging_tiles_m = static_cast<int>((M + gws::STAGING - 1) / gws::STAGING);
  p.staging_tiles_n = static_cast<int>(stn);
  p.alpha = alpha;
  p.beta = beta;
  p.has_c = beta != 0.0f ? 1 : 0;
  p.wide_d = wide_d ? 1 : 0;
  p.streamout = staging ? 1 : 0;
  p.flags = flags;
  p.counter = h->work;
  p.status = h->work + 1;
  p.done = h->work + 2;
  p.timeout_ns = h->timeout_ns;
#ifdef GEMM_WS_DEBUG
  p.debug_fault = h->debug_fault;
  p.trace = h->trace;
  p.phases = h->phases;
#endif

  cudaError_t e;
  {
    // Programmatic stream serialisation: this grid may be scheduled while the
    // previous kernel in the stream finishes; it waits for that kernel before
    // its first global-memory access (grid_dependency_wait in the kernel).
    const int64_t clusters = q.clusters;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (h->pdl) {
      attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[nattr].val.programmaticStreamSerializationAllowed = 1;
      ++nattr;
    }
    if (cs > 1) {
      attr[nattr].id = cudaLaunchAttributeClusterDimension;
      attr[nattr].val.clusterDim.x = cs;
      attr[nattr].val.clusterDim.y = 1;
      attr[nattr].val.clusterDim.z = 1;
      ++nattr;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(cs * clusters), 1, 1);
    cfg.blockDim = dim3(gws::NUM_THREADS, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    if (cg == 1) {
      cfg.dynamicSmemBytes = gws::Cfg<1>::SMEM_BYTES;
      e = cudaLaunchKernelEx(&cfg, gws::gemm_ws_kernel<1>, p);
    } else {
      cfg.dynamicSmemBytes = gws::Cfg<2>::SMEM_BYTES;
      e = cudaLaunchKernelEx(&cfg, gws::gemm_ws_kernel<2>, p);
    }
  }
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (q.sk_first < q.num_tiles && !q.sk_inline) {
    // The split tiles' pieces left fp32 partials; the reduction kernel adds
    // them and writes those tiles' D, next on the same stream.
    gws::ReduceParams rp;
    std::memset(&rp, 0, sizeof rp);
    rp.partial = h->partial;
    rp.C = beta != 0.0f ? C : nullptr;
    rp.D = D;
    rp.M = p.M;
    rp.N = p.N;
    rp.tiles_m = p.tiles_m;
    rp.tiles_n = p.tiles_n;
    rp.group_m = p.group_m;
    rp.cs = cs;
    rp.sk_first = p.sk_first;
    rp.sk_tiles = static_cast<int>(q.num_tiles - q.sk_first);
    rp.sk_split = p.sk_split;
    rp.alpha = alpha;
    rp.beta = beta;
    rp.has_c = p.has_c;
    const int64_t chunks = static_cast<int64_t>(rp.sk_tiles) * cs * 4 * gws::SUB_PER_PART;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(chunks), 1, 1);   // one block per 32 x 32 chunk
    cfg.blockDim = dim3(gws::REDUCE_THREADS, 1, 1);
    cfg.stream = stream;
    if (h->pdl) {
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, gws::gemm_ws_reduce_kernel, rp);
    if (e != cudaSuccess) return cuda_fail(h, e);
  }
  return GEMM_WS_OK;
}

// GEMM_WS_PDL=0 launches without programmatic dependent launch (default on).
int pdl_from_env() {
  if (const char* s = std::getenv("GEMM_WS_PDL")) {
    if (std::atoi(s) == 0) return 0;
  }
  return 1;
}

// GEMM_WS_CTA_GROUP=1 forces single-CTA 128 x 256 tiles, =2 CTA-pair
// 256 x 256 tiles; by default the library picks per problem.
int cta_group_from_env() {
  if (const char* s = std::getenv("GEMM_WS_CTA_GROUP")) {
    const int v = std::atoi(s);
    if (v == 1 || v == 2) return v;
  }
  return 0;
}

// GEMM_WS_STREAM_K: 0 keeps every tile's K range whole; 2 uses stream-K
// wherever the schedule allows it (tests); default 1: where the host cost
// model expects a gain.
int stream_k_from_env() {
  if (const char* s = std::getenv("GEMM_WS_STREAM_K")) {
    const int v = std::atoi(s);
    if (v == 0 || v == 2) return v;
  }
  return 1;
}

// GEMM_WS_SK_INLINE=0 fixes two-piece tiles up with the reduction kernel, as
// tiles of more pieces always are; default 1: inside the GEMM.
int sk_inline_from_env() {
  if (const char* s = std::getenv("GEMM_WS_SK_INLINE")) return std::atoi(s) == 0 ? 0 : 1;
  return 1;
}

// Every other unit of a cluster walks K backwards (default; GEMM_WS_K_SNAKE=0
// turns it off): the clusters' units of one wave run side by side, so each
// wave starts on the A/B k-slices the previous wave loaded last, while L2
// still holds them. Measured at 8192^3: DRAM reads 1.24 -> 1.07 GB per launch,
// time unchanged within noise (interleaved: 8192^3 -0.6 %, 4096^3 -0.3 %,
// 8192 x 8192 x 4096 +0.2 %, ragged batched +1.2 %).
int k_snake_from_env() {
  if (const char* s = std::getenv("GEMM_WS_K_SNAKE")) return std::atoi(s) == 0 ? 0 : 1;
  return 1;
}

// GEMM_WS_GROUP_M overrides the raster group (m-tiles per n step; default 8).
int group_m_from_env() {
  if (const char* s = std::getenv("GEMM_WS_GROUP_M")) {
    const int g = std::atoi(s);
    if (g >= 1 && g <= 1024) return g;
  }
  return 8;
}

class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
    if (prev_ != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
  }

 private:
  int prev_ = -1;
};

}  // namespace

extern "C" {

int gemm_ws_create(gemm_ws_t** out, int device) {
  if (!out) return GEMM_WS_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return GEMM_WS_ERR_CUDA;
  if (device < 0 || device >= count) return GEMM_WS_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return GEMM_WS_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return GEMM_WS_ERR_UNSUPPORTED;

  gemm_ws* h = static_cast<gemm_ws*>(std::calloc(1, sizeof(gemm_ws)));
  if (!h) return GEMM_WS_ERR_CUDA;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->timeout_ns = 1000000000ull;   // 1 s per wait
  if (const char* s = std::getenv("GEMM_WS_TIMEOUT_MS")) {
    const long long ms = std::atoll(s);
    if (ms > 0) h->timeout_ns = static_cast<unsigned long long>(ms) * 1000000ull;
  }

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    std::free(h);
    return GEMM_WS_ERR_CUDA;
  }
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);

  h->cta_group = cta_group_from_env();
  h->pdl = pdl_from_env();
  h->group_m = group_m_from_env();
  h->stream_k = stream_k_from_env();
  h->sk_inline = sk_inline_from_env();
  h->k_snake = k_snake_from_env();
  e = configure_kernels(h->num_sms, &h->max_pair_clusters);
  if (e == cudaSuccess && h->max_pair_clusters < 1) h->cta_group = 1;
  const size_t wbytes = work_words(h->num_sms) * sizeof(uint32_t);
  if (e == cudaSuccess) e = cudaMalloc(&h->work, wbytes);
  if (e == cudaSuccess) e = cudaMemset(h->work, 0, wbytes);
  // Stream-K workspace: one 128 x 256 fp32 partial per SM.
  if (e == cudaSuccess)
    e = cudaMalloc(&h->partial, static_cast<size_t>(h->num_sms) * kPartBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    if (h->work) cudaFree(h->work);
    if (h->partial) cudaFree(h->partial);
    std::free(h);
    return GEMM_WS_ERR_CUDA;
  }
  *out = h;
  return GEMM_WS_OK;
}

int gemm_ws_destroy(gemm_ws_t* h) {
  if (!h) return GEMM_WS_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->work);
  cudaFree(h->partial);
  std::free(h);
  return GEMM_WS_OK;
}

int gemm_ws_run(gemm_ws_t* h, const uint16_t* A, const uint16_t* B, const uint16_t* C,
                uint16_t* D, int64_t M, int64_t N, int64_t K, int64_t L, float alpha,
                float beta, void* stream) {
  int rc = check_problem(h, A, B, C, D, M, N, K, L, beta);
  if (rc != GEMM_WS_OK || M * N * L == 0) return rc;
  DeviceGuard guard(h->device);
  return launch(h, A, B, C, D, M, N, K, L, alpha, beta, nullptr, nullptr,
                static_cast<cudaStream_t>(stream));
}

int gemm_ws_run_streamout(gemm_ws_t* h, const uint16_t* A, const uint16_t* B,
                          const uint16_t* C, uint16_t* D, int64_t M, int64_t N, int64_t K,
                          int64_t L, float alpha, float beta, uint16_t* staging,
                          uint32_t* flags, void* stream) {
  int rc = check_problem(h, A, B, C, D, M, N, K, L, beta);
  if (rc != GEMM_WS_OK || M * N * L == 0) return rc;
  if (!staging || !flags) return GEMM_WS_ERR_INVALID_ARG;
  if (!aligned16(staging) || (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return GEMM_WS_ERR_ALIGNMENT;
  const int64_t T = gemm_ws_streamout_tiles(M, N, L);
  const int64_t sbytes = T * gws::STAGING * gws::STAGING * 2, fbytes = 2 * T * 4;
  const int64_t dbytes = 2 * L * M * N;
  if (overlaps(staging, sbytes, flags, fbytes) || overlaps(staging, sbytes, D, dbytes) ||
      overlaps(flags, fbytes, D, dbytes) ||
      (K > 0 && (overlaps(staging, sbytes, A, 2 * L * M * K) ||
                 overlaps(staging, sbytes, B, 2 * L * N * K) ||
                 overlaps(flags, fbytes, A, 2 * L * M * K) ||
                 overlaps(flags, fbytes, B, 2 * L * N * K))) ||
      (beta != 0.0f && (overlaps(staging, sbytes, C, dbytes) || overlaps(flags, fbytes, C, dbytes))))
    return GEMM_WS_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  return launch(h, A, B, C, D, M, N, K, L, alpha, beta, staging, flags,
                static_cast<cudaStream_t>(stream));
}

int gemm_ws_query_status(gemm_ws_t* h, void* stream) {
  if (!h) return GEMM_WS_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e);
  uint32_t st = 0;
  e = cudaMemcpy(&st, h->work + 1, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (st != 0) {
    // Clear the status word, and the stream-out counters and fix-up words
    // in case an aborted launch left them part-way, so the next launch
    // starts from zero. The clear goes on `s` and is waited for, so it is
    // complete before this returns whatever stream the next run uses.
    e = cudaMemsetAsync(h->work, 0, work_words(h->num_sms) * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e);
  }
  return static_cast<int>(st);
}

int gemm_ws_last_cuda_error(gemm_ws_t* h) { return h ? h->last_cuda_error : 0; }

const char* gemm_ws_status_string(int status) {
  switch (status) {
    case GEMM_WS_OK: return "ok";
    case GEMM_WS_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_WS_ERR_ALIGNMENT: return "misaligned pointer or row pitch";
    case GEMM_WS_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case GEMM_WS_ERR_CUDA: return "CUDA error";
    case GEMM_WS_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

#ifdef GEMM_WS_DEBUG
int gemm_ws_debug_configure(gemm_ws_t* h, int fault, unsigned long long* trace) {
  if (!h || fault < 0 || fault > 2) return GEMM_WS_ERR_INVALID_ARG;
  h->debug_fault = fault;
  h->trace = trace;
  return GEMM_WS_OK;
}

int gemm_ws_debug_phases(gemm_ws_t* h, unsigned long long* phases) {
  if (!h) return GEMM_WS_ERR_INVALID_ARG;
  h->phases = phases;
  return GEMM_WS_OK;
}

int gemm_ws_debug_launch_shape(gemm_ws_t* h, int64_t M, int64_t N, int64_t K, int64_t L,
                               int streamout, int* ctas_per_cluster, int* clusters,
                               int* num_units, int* sk_tiles, int* sk_pieces, int* sk_inline) {
  if (!h || !ctas_per_cluster || !clusters || !num_units || !sk_tiles || M <= 0 || N <= 0 ||
      K < 0 || L <= 0)
    return GEMM_WS_ERR_INVALID_ARG;
  const Plan q = make_plan(h, M, N, K, L, streamout != 0);
  *ctas_per_cluster = q.cs;
  *num_units = static_cast<int>(q.num_units);
  *clusters = static_cast<int>(q.clusters);
  *sk_tiles = static_cast<int>(q.num_tiles - q.sk_first);
  if (sk_pieces) *sk_pieces = static_cast<int>(q.sk_split);
  if (sk_inline) *sk_inline = q.sk_inline ? 1 : 0;
  return GEMM_WS_OK;
}

int gemm_ws_debug_schedule(int cta_group, int num_sms, int max_clusters, int stream_k,
                           int64_t M, int64_t N, int64_t K, int64_t L, int streamout, int* rows,
                           int64_t max_rows, int64_t* num_rows, int* plan) {
  if (cta_group < 0 || cta_group > 2 || num_sms < 1 || max_clusters < 1 || !num_rows || !plan ||
      M <= 0 || N <= 0 || K < 0 || L <= 0 || stream_k < 0 || stream_k > 2)
    return GEMM_WS_ERR_INVALID_ARG;
  gemm_ws h;
  std::memset(&h, 0, sizeof h);
  h.num_sms = num_sms;
  h.cta_group = cta_group;
  h.max_pair_clusters = max_clusters;
  if (h.cta_group == 1) h.num_sms = max_clusters;
  h.group_m = 8;
  h.stream_k = stream_k;
  h.sk_inline = 1;
  float dummy = 0.0f;
  h.partial = &dummy;   // only tested for null by the plan
  const Plan q = make_plan(&h, M, N, K, L, streamout != 0);
  gws::Params p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.L = static_cast<int>(L);
  p.tiles_m = static_cast<int>(q.tiles_m);
  p.tiles_n = static_cast<int>(q.tiles_n);
  p.num_tiles = static_cast<int>(q.num_tiles);
  p.num_full = static_cast<int>(q.num_full);
  p.split = static_cast<int>(q.split);
  p.num_units = static_cast<int>(q.num_units);
  p.num_stages = static_cast<int>(q.num_stages);
  p.sk_first = static_cast<int>(q.sk_first);
  p.sk_split = static_cast<int>(q.sk_split);
  p.group_m = h.group_m;
  plan[0] = q.cs;
  plan[1] = static_cast<int>(q.clusters);
  plan[2] = static_cast<int>(q.num_units);
  plan[3] = static_cast<int>(q.num_tiles);
  plan[4] = static_cast<int>(q.num_stages);
  plan[5] = static_cast<int>(q.sk_first);
  plan[6] = static_cast<int>(q.sk_clusters);
  plan[7] = static_cast<int>(q.tiles_m);
  plan[8] = static_cast<int>(q.tiles_n);
  int64_t n = 0;
  const int clusters = static_cast<int>(q.clusters);
  for (int c = 0; c < clusters; ++c) {
    gws::Unit w;
    for (int i = 0; gws::next_unit(p, c, clusters, i, w); ++i) {
      if (rows && n < max_rows) {
        int* r = rows + n * kScheduleCols;
        r[0] = c;
        r[1] = i;
        r[2] = w.id;
        r[3] = w.tile;
        r[4] = w.mb;
        r[5] = w.n0;
        r[6] = w.width;
        r[7] = w.l;
        r[8] = w.kb0;
        r[9] = w.kb1;
        r[10] = w.piece;
        r[11] = w.pieces;
        r[12] = w.sk_tile;
        r[13] = w.first_cluster;
        r[14] = w.pieces > 1 ? gws::sk_slot(p, w, w.piece) : -1;
      }
      ++n;
    }
  }
  *num_rows = n;
  return GEMM_WS_OK;
}
#endif

int64_t gemm_ws_streamout_tiles(int64_t M, int64_t N, int64_t L) {
  if (M <= 0 || N <= 0 || L <= 0) return 0;
  return L * ((M + gws::STAGING - 1) / gws::STAGING) * ((N + gws::STAGING - 1) / gws::STAGING);
}

int gemm_ws_kernels_per_run(gemm_ws_t* h, int64_t M, int64_t N, int64_t K, int64_t L,
                            int streamout) {
  if (!h) return -GEMM_WS_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || L < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim ||
      L > kMaxDim)
    return -GEMM_WS_ERR_INVALID_ARG;
  if (M * N * L == 0) return 0;
  const Plan q = make_plan(h, M, N, K, L, streamout != 0);
  return q.sk_first < q.num_tiles && !q.sk_inline ? 2 : 1;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free stream-out entry point.
//
// For callers that must not allocate device memory themselves or through the
// library: code running where cudaMalloc is unavailable or forbidden (inside
// another allocator's callback, under a framework that owns every device
// allocation and pools it, or in a process that reserved all memory up
// front). gemm_ws_create needs cudaMalloc for its workspace; this entry point
// needs no handle. Its only scratch (the stream-out sequence counter and the
// watchdog status word) lives in the fixed array below, which every GPU that
// loads this library holds until the process exits.

namespace {

constexpr int kNoAllocScratchWords = 64;   // 256 bytes per device; 2 words used
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  bool ready;
  int num_sms;
  int cta_group;
  int max_pair_clusters;
  uint32_t* scratch;   // device address of g_noalloc_scratch on this device
  unsigned long long timeout_ns;
  PFN_cuTensorMapEncodeTiled_v12000 encode;
#ifdef GEMM_WS_DEBUG
  int debug_fault;                      // set by gemm_ws_debug_noalloc_configure
  unsigned long long debug_timeout_ns;  // 0: timeout_ns
#endif
};

NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

}  // namespace

// word 0: stream-out sequence counter, word 1: watchdog status, word 2:
// consumer warps finished (the kernel returns words 0 and 2 to zero).
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

namespace {

// Once per device, with that device current: checks it is sm_103, reads its
// SM count, sets the kernel's shared-memory attribute, fetches the tensor-map
// encoder and takes the device address of the scratch array. Allocates
// nothing.
int noalloc_setup(int device, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice& d = g_noalloc_devices[device];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return GEMM_WS_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_WS_ERR_UNSUPPORTED;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return GEMM_WS_ERR_CUDA;
    int pair_clusters = 0;
    if (configure_kernels(sms, &pair_clusters) != cudaSuccess) return GEMM_WS_ERR_CUDA;
    d.cta_group = pair_clusters >= 1 ? cta_group_from_env() : 1;
    d.max_pair_clusters = pair_clusters;
    uint32_t* ptr = nullptr;
    // In host code the array's name is only a host-side stand-in; the kernel
    // must be given this device address instead.
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess ||
        !ptr)
      return GEMM_WS_ERR_CUDA;
    d.timeout_ns = 1000000000ull;
    if (const char* s = std::getenv("GEMM_WS_TIMEOUT_MS")) {
      const long long ms = std::atoll(s);
      if (ms > 0) d.timeout_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    d.num_sms = sms;
    d.scratch = ptr;
    d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    d.ready = true;
  }
  *out = &d;
  return GEMM_WS_OK;
}

}  // namespace

extern "C" int gemm_ws_run_streamout_noalloc(const uint16_t* A, const uint16_t* B,
                                             const uint16_t* C, uint16_t* D, int64_t M,
                                             int64_t N, int64_t K, int64_t L, float alpha,
                                             float beta, uint16_t* staging, uint32_t* flags,
                                             void* stream) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return GEMM_WS_ERR_CUDA;
  if (device < 0 || device >= kNoAllocMaxDevices) return GEMM_WS_ERR_INVALID_ARG;
  // The sequence counter in the scratch numbers tiles with 31 bits.
  if (gemm_ws_streamout_tiles(M, N, L) > kMaxDim) return GEMM_WS_ERR_INVALID_ARG;
  NoAllocDevice* d = nullptr;
  int rc = noalloc_setup(device, &d);
  if (rc != GEMM_WS_OK) return rc;
  gemm_ws h;   // a handle on the host stack that borrows the static scratch
  std::memset(&h, 0, sizeof h);
  h.device = device;
  h.num_sms = d->num_sms;
  h.cta_group = d->cta_group;
  h.pdl = pdl_from_env();
  h.group_m = group_m_from_env();
  h.k_snake = k_snake_from_env();   // same schedule, hence same bits, as a handle
  h.max_pair_clusters = d->max_pair_clusters;
  h.work = d->scratch;
  h.timeout_ns = d->timeout_ns;
  h.encode = d->encode;
#ifdef GEMM_WS_DEBUG
  h.debug_fault = d->debug_fault;
  if (d->debug_timeout_ns) h.timeout_ns = d->debug_timeout_ns;
#endif
  return gemm_ws_run_streamout(&h, A, B, C, D, M, N, K, L, alpha, beta, staging, flags, stream);
}

#ifdef GEMM_WS_DEBUG
extern "C" int gemm_ws_debug_noalloc_configure(int device, int fault, long long timeout_ms) {
  if (device < 0 || device >= kNoAllocMaxDevices || fault < 0 || fault > 1 || timeout_ms < 0)
    return GEMM_WS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice& d = g_noalloc_devices[device];
  d.debug_fault = fault;
  d.debug_timeout_ns = static_cast<unsigned long long>(timeout_ms) * 1000000ull;
  return GEMM_WS_OK;
}
#endif

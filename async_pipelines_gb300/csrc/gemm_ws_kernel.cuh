// Persistent warp-specialized bf16 GEMM for GB300 (sm_103a), one CTA per SM.
//
//   D[l] = alpha * A[l] * B[l] + beta * C[l]     (fp32 accumulate in TMEM)
//
// Warp roles (the SM90 cooperative kernel's producer / consumer / epilogue
// split of "sm90_gemm_tma_warpspecialized_cooperative.hpp", re-cut for
// tcgen05, whose accumulators live in tensor memory instead of registers):
//   warps 0, 11  TMA producers (A loads, B loads): fill a STAGES-deep
//              shared-memory ring of A/B k-blocks guarded by full/empty
//              mbarriers; warp 0 is the task leader that arms full[s]. Like the
//              SM100 mainloop `load()` discussed in "why does load() pre-issue
//              producer_try_acquire", each probes the NEXT stage's empty
//              barrier (non-blocking token) before issuing the current copies.
//   warp 1     MMA issuer: one thread issues tcgen05.mma (N = 256, K = 16)
//              into one of two TMEM accumulators and releases each stage with
//              tcgen05.commit -> empty[s]; a tile's last commit -> acc_full.
//   warps 2-9  epilogue: two warps per 32-lane quarter of TMEM (rows), each
//              draining alternate 32-column subtiles TMEM -> registers, applies
//              alpha/beta (C arrives by TMA), rounds to bf16, writes a
//              swizzled shared-memory slot and TMA-stores it to D over a
//              two-slot store pipeline (bulk-group read waits), as in the
//              Hopper epilogue loop quoted in "How to build a pipeline between
//              epilogue and communication warp groups?".
//   warp 10    stream-out consumer (optional): the per-tile handoff that issue
//              asks for. The epilogue arrives on d_full[slot] after writing a
//              slot; the consumer waits on it, copies the slot into a packed
//              staging buffer with its own TMA store, waits for that store's
//              shared-memory reads, and arrives on d_empty[slot]. The epilogue
//              reuses a slot only after BOTH its own bulk-group read wait and
//              d_empty, which is the answer to the issue's problem that bulk
//              groups are per thread and invisible to another warp.
//
// CTA group CG (template parameter):
//   CG == 1  one CTA computes a 128 x 256 tile (tcgen05.mma.cta_group::1,
//            M = 128); it loads a 128 x 64 slab of A and a 256 x 64 slab of B
//            per k-block.
//   CG == 2  a cluster of two CTAs computes a 256 x 256 tile with
//            tcgen05.mma.cta_group::2 (M = 256) issued by the even CTA only;
//            each CTA loads its own 128 rows of A and its own 128 rows of B
//            (128 x 64 each, no multicast), and each CTA's TMEM receives its
//            128 rows of D. The TMA of both CTAs completes on the even CTA's
//            full[s] barrier, which the even producer arms for both; the MMA's
//            commits are multicast to both CTAs' empty / acc_full barriers;
//            the epilogue warps of both CTAs release acc_empty on the even
//            CTA. This is the CTA-pair pipeline of the CuTe DSL pipeline page
//            (UMMA commits per CTA group, async producers signalling the even
//            CTA of the pair).
//
// Every role walks the same static persistent unit sequence (next_unit:
// cluster c takes tiles c, c + #clusters, ..., and, where the host planned
// it, one equal piece of a tile's K range as its last unit), so the
// scheduler needs no communication. The pieces of a tile leave fp32 partials
// in a workspace, which gemm_ws_reduce_kernel adds after the GEMM (the
// separate-reduction form of the SM90 cooperative kernel's fix-up). Every
// wait is bounded by a watchdog (global timer): on expiry the kernel records
// GEMM_WS_ERR_TIMEOUT in a status word, all roles leave their loops,
// in-flight copies are drained and TMEM is freed.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gws {

constexpr int BM = 128;                  // rows per CTA = TMEM lanes
constexpr int BN = 256;                  // tile columns (UMMA N)
constexpr int BK = 64;                   // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;               // K of one tcgen05.mma kind::f16
constexpr int ACC_BUFS = 2;              // TMEM accumulators (MMA overlaps epilogue)
constexpr int EPI_N = 32;                // columns per epilogue subtile
constexpr int EPI_SLOTS = 2;             // D shared-memory slots when C is read
constexpr int EPI_SLOTS_NOC = 4;         // ... when it is not (the C buffers become D slots)
constexpr int NUM_EPI_WARPS = 8;         // two per TMEM lane quarter
constexpr int EPI_HALF_WARPS = 4;        // one per lane quarter: a half covers 128 rows
constexpr int STAGING = 128;             // stream-out tile edge
constexpr int SUB_PER_STAGING = STAGING / EPI_N;
constexpr int SUB_PER_PART = BN / EPI_N;   // subtiles (32 x 32 chunks per lane quarter) of a part
constexpr int CHUNK_FLOATS = 32 * EPI_N;      // one 32 x 32 fp32 partial chunk
constexpr uint32_t CHUNK_BYTES = CHUNK_FLOATS * 4;
// A piece's partial, per epilogue warp (lane quarter q, subtiles j = hf + 2k):
// the warp's four chunks k = 0..3 lie together, so that one bulk copy moves
// them; chunk (q, j) of a CTA's part starts at this many floats.
__host__ __device__ __forceinline__ int part_chunk_offset(int q, int j) {
  return ((q * 2 + (j & 1)) * 4 + (j >> 1)) * CHUNK_FLOATS;
}
constexpr int PART_FLOATS = 4 * SUB_PER_PART * CHUNK_FLOATS;   // a CTA's 128 x 256 partial
constexpr int WARP_TMA = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_EPI0 = 2;
constexpr int WARP_CONSUMER = WARP_EPI0 + NUM_EPI_WARPS;
constexpr int WARP_TMA_B = WARP_CONSUMER + 1;   // second producer warp: the B loads
constexpr int NUM_THREADS = (WARP_TMA_B + 1) * 32;
constexpr uint32_t TMEM_COLS = ACC_BUFS * BN;   // 512: all of the SM's TMEM
constexpr uint32_t A_SLAB_BYTES = BM * BK * 2;           // 16 KiB: 128 x 64 slab of A
constexpr uint32_t EPI_QUARTER_BYTES = 32 * EPI_N * 2;   // 2 KiB: one warp's rows
constexpr uint32_t EPI_SLOT_BYTES = BM * EPI_N * 2;      // 8 KiB: 128 rows
constexpr uint32_t WIDE_QUARTER_BYTES = 32 * 2 * EPI_N * 2;   // 4 KiB: 32 x 64 block of D
constexpr uint32_t STATUS_TIMEOUT = 5;   // == GEMM_WS_ERR_TIMEOUT
constexpr uint32_t WAIT_HINT_NS = 1000000;   // suspend bound of one try_wait

// barrier indices
constexpr int NUM_STAGES_MAX = 6;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + NUM_STAGES_MAX;
constexpr int BAR_ACC_FULL = BAR_EMPTY + NUM_STAGES_MAX;
constexpr int BAR_ACC_EMPTY = BAR_ACC_FULL + ACC_BUFS;
constexpr int BAR_C_FULL = BAR_ACC_EMPTY + ACC_BUFS;          // [epilogue warp]
constexpr int BAR_D_FULL = BAR_C_FULL + NUM_EPI_WARPS;
constexpr int BAR_D_EMPTY = BAR_D_FULL + EPI_SLOTS_NOC;
constexpr int BAR_MMA_DRAIN = BAR_D_EMPTY + EPI_SLOTS_NOC;
constexpr int BAR_FIX = BAR_MMA_DRAIN + 1;                      // [epilogue warp][chunk]
constexpr int NUM_BARS = BAR_FIX + NUM_EPI_WARPS * 4;

template <int CG>
struct Cfg {
  static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
  static constexpr int CS = CG;                          // CTAs per cluster
  static constexpr int TILE_M = BM * CG;                 // rows per (pair) tile
  static constexpr int B_ROWS = BN / CG;                 // B rows in each CTA's stage
  static constexpr uint16_t ALL_CTAS = static_cast<uint16_t>((1u << CS) - 1u);
  // 64-deep k-blocks per ring stage. The CTA pair takes two (a 128-deep
  // stage of 64 KiB, 3 stages): half the barrier round trips per MMA, which
  // measured ~10 % more tensor throughput per clock than 6 stages of 64.
  static constexpr int KSUB = CG == 1 ? 1 : 2;
  static constexpr int STAGES = CG == 1 ? 4 : 3;
  static constexpr uint32_t A_BLOCK_BYTES = A_SLAB_BYTES;        // one 128 x 64 slab
  static constexpr uint32_t B_BLOCK_BYTES = B_ROWS * BK * 2;      // one B_ROWS x 64 slab
  static constexpr uint32_t A_BYTES = KSUB * A_BLOCK_BYTES;       // A part of a stage
  static constexpr uint32_t B_STAGE_BYTES = KSUB * B_BLOCK_BYTES; // B part of a stage
  static constexpr uint32_t STAGE_TX = CG * (A_BYTES + B_STAGE_BYTES);
  static constexpr uint32_t STAGE_TX_HALF = CG * (A_BYTES + B_STAGE_BYTES / 2);
  static constexpr uint32_t STAGE_TX_QUARTER = CG * (A_BYTES + B_STAGE_BYTES / 4);
  // Shared-memory carve-out (offsets from a 1024-byte aligned base).
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
  // Epilogue region: D slots 0-1, then either the C buffers (beta != 0) or
  // D slots 2-3 (beta == 0); slot s sits at OFF_D + s * EPI_SLOT_BYTES.
  static constexpr uint32_t OFF_D = OFF_B + STAGES * B_STAGE_BYTES;
  static constexpr uint32_t OFF_C = OFF_D + EPI_SLOTS * EPI_SLOT_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_C + NUM_EPI_WARPS * EPI_QUARTER_BYTES;
  static_assert(EPI_SLOTS_NOC * EPI_SLOT_BYTES == OFF_BAR - OFF_D, "epilogue region");
  static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + slack to align the base
  static constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, BN);
  static constexpr uint32_t IDESC_HALF = idesc_bf16_f32(TILE_M, BN / 2);
  static constexpr uint32_t IDESC_QUARTER = idesc_bf16_f32(TILE_M, BN / 4);
  static_assert(STAGES <= NUM_STAGES_MAX, "barrier table");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB per-CTA shared memory");
  static_assert(OFF_B % 1024 == 0 && OFF_D % 1024 == 0 && OFF_C % 1024 == 0, "alignment");
};

struct Params {
  CUtensorMap tmA;   // {K, M, L}, box {64, 128}, 128-byte swizzle
  CUtensorMap tmB;   // {K, N, L}, box {64, 256 / CG}, 128-byte swizzle
  CUtensorMap tmB2;  // {K, N, L}, box {64, 128 / CG}: B of a half-width unit
  CUtensorMap tmB4;  // {K, N, L}, box {64, 64 / CG}: B of a quarter-width unit
  CUtensorMap tmC;   // {N, M, L}, box {32, 32},  64-byte swizzle (beta != 0)
  CUtensorMap tmD;   // {N, M, L}, box {32, 32},  64-byte swizzle
  CUtensorMap tmDw;  // {N, M, L}, box {64, 32}, 128-byte swizzle (wide stores)
  CUtensorMap tmS;   // staging {128, 128, T}, box {32, 128}, 64-byte swizzle
  int M, N, K, L;
  int tiles_m, tiles_n, num_tiles, num_kb;   // tiles of 128*CG x 256
  int num_full;                  // tiles [0, num_full) run whole; the rest as `split` parts
  int split;                     // 2: halves (128 columns), 4: quarters (64 columns)
  int num_units;                 // work units (see unit_coords)
  int num_stages;                // ring stages covering K (KSUB k-blocks each)
  // Stream-K: the K ranges of tiles [sk_first, num_tiles) are cut into
  // sk_split equal pieces; sk_first == num_tiles: none.
  int sk_first;
  int sk_split;
  float* partial;                // piece partials: [cluster][CTA][chunk] x 1024 fp32
  // In-kernel fix-up of two-piece tiles (sk_inline, sk_split == 2): per
  // epilogue warp of each CTA, an arrival count per split tile and a
  // partial-written flag per piece (see sk_arrival_word / sk_written_word);
  // all zero at launch, and the kernel leaves them zero again.
  int sk_inline;
  uint32_t* sk_sync;
  int group_m;                   // raster: tiles walk group_m m-tiles per n step
  int k_snake;                   // 1: every other unit of a cluster walks K backwards
  int staging_tiles_m;           // ceil(M / 128)
  int staging_tiles_n;           // ceil(N / 128)
  float alpha, beta;
  int has_c;                     // beta != 0
  int wide_d;                    // D stores in 32 x 64 blocks (beta == 0, no stream-out,
                                 // no split pieces, short K)
  int streamout;
  uint32_t* flags;               // 2 * T words (stream-out)
  uint32_t* counter;             // stream-out sequence counter (zero at launch; the
                                 // kernel's last consumer warp zeroes it again)
  uint32_t* done;                // consumer warps finished (same life cycle)
  uint32_t* status;              // watchdog status word
  unsigned long long timeout_ns; // bound of every single wait
#ifdef GEMM_WS_DEBUG
  int debug_fault;               // 1: the stream-out consumer takes no tile; 2: split pieces
                                 // never flag their written partial
  unsigned long long* trace;     // [tile][CG][2] global-timer stamps, or null
  unsigned long long* phases;    // [CTA][8] stamps (see gemm_ws_debug_phases), or null
#endif
};

// Tile t -> (m block, n block, batch). Within a batch, tiles go down a group
// of `group_m` m-blocks, then step n, so the CTAs resident at one time share
// their A rows and B columns through L2.
__host__ __device__ __forceinline__ void tile_coords_of(int tiles_m, int tiles_n, int group_m,
                                                        int t, int& mb, int& nb, int& l) {
  const int per_batch = tiles_m * tiles_n;
  l = t / per_batch;
  const int r = t - l * per_batch;
  const int group_tiles = group_m * tiles_n;
  const int g = r / group_tiles;
  const int first_m = g * group_m;
  const int gm = tiles_m - first_m < group_m ? tiles_m - first_m : group_m;
  const int rr = r - g * group_tiles;
  mb = first_m + rr % gm;
  nb = rr / gm;
}

__host__ __device__ __forceinline__ void tile_coords(const Params& p, int t, int& mb, int& nb, int& l) {
  tile_coords_of(p.tiles_m, p.tiles_n, p.group_m, t, mb, nb, l);
}

// A unit of work: a tile (256 columns, or, for the last tiles in raster
// order, one 128-column half, so that the final wave of the persistent
// schedule is not left half idle; or, in a problem of so few tiles that four
// units per tile fit on the GPU at once, one 64-column quarter), or a piece
// of a tile's K range.
struct Unit {
  int mb, l;
  int n0;      // first column
  int width;   // 256, 128 or 64 columns
  int tile;    // tile index
  int kb0, kb1;        // ring stages [kb0, kb1) of the tile's K range
  int piece, pieces;   // piece `piece` of the `pieces` that share the K range (1: whole)
  int sk_tile;         // index in the stream-K region
  int first_cluster;   // cluster that runs piece 0 (piece k runs on first_cluster + k)
  int id;              // unit number (trace index)
  int rev;             // the producer walks the k range from its end
};

__host__ __device__ __forceinline__ Unit whole_tile(const Params& p, int t) {
  Unit w;
  int nb;
  tile_coords(p, t, w.mb, nb, w.l);
  w.n0 = nb * BN;
  w.width = BN;
  w.tile = t;
  w.kb0 = 0;
  w.kb1 = p.num_stages;
  w.piece = 0;
  w.pieces = 1;
  w.sk_tile = -1;
  w.first_cluster = 0;
  w.id = t;
  w.rev = 0;
  return w;
}

// Without stream-K: unit u < num_full is tile u; the units after it are the
// halves (split == 2) or quarters (split == 4) of the remaining tiles.
__host__ __device__ __forceinline__ Unit unit_coords(const Params& p, int u) {
  if (u < p.num_full) return whole_tile(p, u);
  const int h = u - p.num_full;
  const int lg = p.split == 4 ? 2 : 1;
  Unit w = whole_tile(p, p.num_full + (h >> lg));
  w.width = BN >> lg;
  w.n0 += (h & (p.split - 1)) * w.width;
  w.id = u;
  return w;
}

// Workspace slot of piece k of a stream-K tile: the cluster that runs it.
__host__ __device__ __forceinline__ int sk_slot(const Params&, const Unit& w, int k) {
  return w.first_cluster + k;
}

// In-kernel fix-up words of epilogue warp e of CTA `rank` (cs CTAs per
// cluster): the arrival count of split tile r (its sk_tile), then the flag
// that the piece in workspace slot s has written its partial. Each area has
// gridDim.x * NUM_EPI_WARPS words (r and s are below the cluster count).
__device__ __forceinline__ uint32_t* sk_arrival_word(const Params& p, int cs, int r,
                                                     uint32_t rank, int e) {
  return p.sk_sync + (static_cast<size_t>(r) * cs + rank) * NUM_EPI_WARPS + e;
}
__device__ __forceinline__ uint32_t* sk_written_word(const Params& p, int cs, int s,
                                                     uint32_t rank, int e) {
  return p.sk_sync + static_cast<size_t>(gridDim.x) * NUM_EPI_WARPS +
         (static_cast<size_t>(s) * cs + rank) * NUM_EPI_WARPS + e;
}

// The i-th unit of cluster c (of `clusters`), in the order every role of the
// cluster walks them; false once the cluster has no more. With a stream-K
// region, every cluster first runs its whole tiles (tile c, c + clusters,
// ...; sk_first is a multiple of clusters), then cluster c = r * S + s (S =
// sk_split) runs piece s of the region's tile r as its last unit: ring stages
// [s * ns / S, (s + 1) * ns / S), a work unit with its own k-tile start and
// count, as in the SM90 cooperative kernel's operator(). Piece s of every
// tile covers the same k range. Every unit's place follows from this
// arithmetic alone, so no role needs to exchange schedule information.
__host__ __device__ __forceinline__ bool next_unit(const Params& p, int c, int clusters, int i, Unit& w) {
  if (p.sk_first >= p.num_tiles) {   // whole tiles, then halves: static stride
    const int u = c + i * clusters;
    if (u >= p.num_units) return false;
    w = unit_coords(p, u);
    w.rev = p.k_snake & i;
    return true;
  }
  const int dp = p.sk_first / clusters;
  if (i < dp) {
    w = whole_tile(p, c + i * clusters);
    w.rev = p.k_snake & i;
    return true;
  }
  const int S = p.sk_split;
  if (i > dp || c >= (p.num_tiles - p.sk_first) * S) return false;
  const int r = c / S, sp = c - r * S;
  const long long ns = p.num_stages;
  w = whole_tile(p, p.sk_first + r);
  w.kb0 = static_cast<int>(sp * ns / S);
  w.kb1 = static_cast<int>((sp + 1) * ns / S);
  w.piece = sp;
  w.pieces = S;
  w.sk_tile = r;
  w.first_cluster = r * S;
  w.id = p.sk_first + c;
  return true;
}

// Stream-out tiles (128 x 128) of this CTA's 128-row part of a unit that
// exist inside M x N: 0, 1 or 2. Epilogue and consumer use the same count.
// (Stream-out launches have no quarter units.)
__device__ __forceinline__ int staging_in_part(const Params& p, int row_tile, const Unit& w) {
  if (row_tile >= p.staging_tiles_m || w.n0 >= p.N) return 0;
  const int cols_left = p.N - w.n0;
  return min(w.width / STAGING, (cols_left + STAGING - 1) / STAGING);
}

// 32-column subtiles the epilogue stores for this CTA's 128-row part of a
// unit: the part's columns inside N, rounded up to whole 128-column blocks
// (the TMA stores clip at N), at most the unit's width: 0, 2, 4 or 8.
__device__ __forceinline__ int subtiles_in_part(const Params& p, int row_tile, const Unit& w) {
  if (row_tile >= p.staging_tiles_m || w.n0 >= p.N) return 0;
  const int cols = ((p.N - w.n0 + STAGING - 1) / STAGING) * STAGING;
  return min(w.width, cols) / EPI_N;
}

struct Watchdog {
  volatile uint32_t* abort;   // shared-memory abort flag of this CTA
  uint32_t* status;           // global status word
  unsigned long long limit_ns;
};

// Bounded wait on an mbarrier phase. The probe may suspend the thread until
// the phase completes (or WAIT_HINT_NS passes), so waiting costs few issue
// slots. Returns false if the CTA is aborting or this wait exceeded the limit
// (which then starts the abort). kCluster selects cluster-scope acquire, for
// barriers that the peer CTA arrives on.
template <bool kCluster>
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  auto probe = [&]() {
    uint32_t ok;
    if (kCluster)
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(bar), "r"(parity), "r"(WAIT_HINT_NS)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(bar), "r"(parity), "r"(WAIT_HINT_NS)
          : "memory");
    return ok != 0;
  };
  if (probe()) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (probe()) return true;
    if (*wd.abort) return false;
    if (global_timer_ns() - t0 > wd.limit_ns) {
      *wd.abort = 1;
      atomicExch(wd.status, STATUS_TIMEOUT);
      return false;
    }
  }
}

// Non-blocking cluster-scope probe.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

template <bool kCluster>
__device__ __noinline__ bool spin_slow(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (kCluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (*wd.abort) return false;
      if (global_timer_ns() - t0 > wd.limit_ns) {
        *wd.abort = 1;
        atomicExch(wd.status, STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait for the latency-critical producer and MMA threads: polls
// without ever suspending, because the wake-up delay of a suspended try_wait
// lands directly on the load -> MMA critical path.
template <bool kCluster>
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  if (kCluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
  return spin_slow<kCluster>(bar, parity, wd);
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_timer_ns() - t0 > 100000000ull) return;   // 100 ms
  }
}

// Warp-uniform wait: lane 0 waits, the verdict is broadcast to the warp.
// On success every lane then probes the (already completed) phase once, so
// each thread itself observes the completion (acquire) before touching the
// data it guards. The phase cannot move on meanwhile: its next completion
// needs an arrival that this warp makes only later.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bounded<true>(bar, parity, wd) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait_cluster(bar, parity);
  __syncwarp();
  return ok != 0;
}

// Warp-uniform wait for the epilogue's short, latency-critical handoffs (C
// arrival, a free D slot): lane 0 polls without suspending.
__device__ __forceinline__ bool warp_wait_spin(uint32_t bar, uint32_t parity,
                                               const Watchdog& wd) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_spin<true>(bar, parity, wd) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait_cluster(bar, parity);
  __syncwarp();
  return ok != 0;
}

// Warp-uniform bounded wait for a flag in global memory that another CTA
// sets with release semantics (the in-kernel fix-up's partial-written flag):
// lane 0 polls with acquire loads; on success every lane loads the flag once
// more with acquire, so each thread itself is ordered after the writer's
// partial stores.
__device__ __noinline__ bool flag_wait_slow(const uint32_t* f, const Watchdog& wd) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_gpu(f) != 0u) return true;
    if ((it & 63) == 0) {
      if (*wd.abort) return false;
      if (global_timer_ns() - t0 > wd.limit_ns) {
        *wd.abort = 1;
        atomicExch(wd.status, STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool warp_wait_flag(const uint32_t* f, const Watchdog& wd) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = (ld_acquire_gpu(f) != 0u || flag_wait_slow(f, wd)) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_gpu(f);
  __syncwarp();
  return ok != 0;
}

// ------------------------------------------------------------ producer

// Two producer warps feed the ring, as the task-leader pipeline of the CuTe DSL
// pipeline page (`TSPipelineTmaAsync`) does: both acquire every empty[s]
// (each waits for the stage to be free before writing into it), warp A loads
// the A slabs and warp B the B slabs, and only warp A — the task leader of
// the even CTA — arms full[s], once, with the byte count of everything that
// lands in the stage (the B bytes may complete before the arming; the phase
// cannot complete before the leader's arrival). Issuing the two operand
// streams from two threads measured 2-3 % more tensor throughput per clock.
enum ProducerPart { LOAD_A = 0, LOAD_B = 1 };

template <int CG>
__device__ __forceinline__ void producer_role(const Params& p, uint32_t sbase, uint32_t rank,
                                              ProducerPart part, const Watchdog& wd) {
  using C = Cfg<CG>;
  auto full = [&](uint32_t s) { return sbase + C::OFF_BAR + 8 * (BAR_FULL + s); };
  auto empty = [&](uint32_t s) { return sbase + C::OFF_BAR + 8 * (BAR_EMPTY + s); };
  const int cluster = blockIdx.x / C::CS, clusters = gridDim.x / C::CS;
  const int h = static_cast<int>(rank);   // CTA of the pair (0: even)
  const bool leader = part == LOAD_A && h == 0;   // arms full[s] for the pair
  uint32_t g = 0;   // stages issued by this warp so far (ring position)
  bool ok = true;
  // The producer starts in the opposite phase: the first STAGES waits on a
  // freshly initialised empty barrier (parity 1) succeed at once.
  bool token = mbar_test_wait(empty(0), 1);
  Unit w;
  for (int it = 0; ok && next_unit(p, cluster, clusters, it, w); ++it) {
    const int l = w.l;
    const int a_row = (w.mb * C::CS + static_cast<int>(rank)) * BM;   // this CTA's rows
    const int b_row = w.n0 + h * (w.width / CG);                      // its half of the N range
    const CUtensorMap* tmb = w.width == BN ? &p.tmB : (w.width == BN / 2 ? &p.tmB2 : &p.tmB4);
    const uint32_t tx = w.width == BN       ? C::STAGE_TX
                        : w.width == BN / 2 ? C::STAGE_TX_HALF
                                            : C::STAGE_TX_QUARTER;
    for (int it = 0; it < w.kb1 - w.kb0; ++it) {
      // With k_snake, odd units walk K from the end, so a wave starts on the
      // k-slices the previous wave loaded last, while L2 still holds them.
      const int kb = w.rev ? w.kb1 - 1 - it : w.kb0 + it;
      const uint32_t s = g % C::STAGES;
      const uint32_t ph = (g / C::STAGES) & 1;
      if (!token && !wait_spin<false>(empty(s), ph ^ 1, wd)) {
        ok = false;
        break;
      }
      ++g;
      // try-acquire the NEXT stage before this stage's copies go out
      token = mbar_test_wait(empty(g % C::STAGES), ((g / C::STAGES) & 1) ^ 1);
      if (g == 1) {
        grid_dependency_wait();   // A and B may be the previous kernel's output
#ifdef GEMM_WS_DEBUG
        if (p.phases && threadIdx.x == 0) p.phases[blockIdx.x * 8 + 1] = global_timer_ns();
#endif
      }
      if (leader) mbar_arrive_expect_tx(full(s), tx);
      // Both CTAs' copies complete on the pair's even CTA's full[s]. Slabs
      // past K (a ragged last stage) are zero-filled by the TMA.
      const uint32_t full_bar = CG == 1 ? full(s) : mapa_shared(full(s), 0u);
#pragma unroll
      for (int ks = 0; ks < C::KSUB; ++ks) {
        const int k0 = (kb * C::KSUB + ks) * BK;
        if (part == LOAD_A) {
          const uint32_t adst = sbase + C::OFF_A + s * C::A_BYTES + ks * C::A_BLOCK_BYTES;
          if constexpr (CG == 1)
            tma_load_3d(adst, &p.tmA, full_bar, k0, a_row, l);
          else
            tma_load_3d_pair(adst, &p.tmA, full_bar, k0, a_row, l);
        } else {
          const uint32_t bdst = sbase + C::OFF_B + s * C::B_STAGE_BYTES + ks * C::B_BLOCK_BYTES;
          if constexpr (CG == 1)
            tma_load_3d(bdst, tmb, full_bar, k0, b_row, l);
          else
            tma_load_3d_pair(bdst, tmb, full_bar, k0, b_row, l);
        }
      }
    }
  }
  if (!ok && leader) {
    // Abort: wait (bounded) for the copies of the last stages armed, so no
    // TMA write lands after the CTA pair has released its shared memory.
    const uint32_t first = g > C::STAGES ? g - C::STAGES : 0;
    for (uint32_t j = first; j < g; ++j) wait_drain(full(j % C::STAGES), (j / C::STAGES) & 1);
  } else if (!ok) {
    // Abort, other producer warps: their last copies may target a stage the
    // leader never armed, so no barrier tracks them; give them 100 us (copies
    // take a few) before the CTA moves on to its exit.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 100000ull) __nanosleep(1000);
  }
}

// ------------------------------------------------------------ MMA issuer

template <int CG>
__device__ __forceinline__ void mma_role(const Params& p, uint32_t sbase, uint32_t tmem_base,
                                         uint32_t rank, const Watchdog& wd) {
  using C = Cfg<CG>;
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8 * i; };
  // Stage releases and accumulator commits go to both CTAs of the pair.
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << rank);
  auto commit = [&](uint32_t b, uint16_t mask) {
    if constexpr (CG == 1)
      umma_commit(b);
    else
      umma_commit_pair(b, mask);
  };
  const int cluster = blockIdx.x / C::CS, clusters = gridDim.x / C::CS;
  uint32_t g = 0;
  int i = 0;
  bool issued = false;
  Unit w;
  for (; next_unit(p, cluster, clusters, i, w); ++i) {
    const uint32_t b = i & 1, aph = (i >> 1) & 1;
    const uint32_t idesc =
        w.width == BN ? C::IDESC : (w.width == BN / 2 ? C::IDESC_HALF : C::IDESC_QUARTER);
    if (!wait_spin<true>(bar(BAR_ACC_EMPTY + b), aph ^ 1, wd)) goto done;
    tc_fence_after_sync();   // epilogue's TMEM reads of buffer b precede these MMAs
    {
      const uint32_t d_tmem = tmem_base + b * BN;
      for (int it = 0; it < w.kb1 - w.kb0; ++it) {   // stages in the order the producer loads them
        const uint32_t s = g % C::STAGES;
        // The stage's bytes are ordered before the MMA by the barrier's
        // transaction count (TMA and tcgen05 both act in the async proxy).
        if (!wait_spin<true>(bar(BAR_FULL + s), (g / C::STAGES) & 1, wd)) goto done;
        const uint32_t a_addr = sbase + C::OFF_A + s * C::A_BYTES;
        const uint32_t b_addr = sbase + C::OFF_B + s * C::B_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::KSUB * (BK / UMMA_K); ++kk) {
          const int blk = kk / (BK / UMMA_K), kin = kk % (BK / UMMA_K);
          const uint64_t ad =
              sdesc_kmajor_sw128(a_addr + blk * C::A_BLOCK_BYTES + kin * UMMA_K * 2);
          const uint64_t bd =
              sdesc_kmajor_sw128(b_addr + blk * C::B_BLOCK_BYTES + kin * UMMA_K * 2);
          const uint32_t acc = (it != 0 || kk != 0) ? 1u : 0u;
          if constexpr (CG == 1)
            umma_bf16(d_tmem, ad, bd, idesc, acc);
          else
            umma_bf16_pair(d_tmem, ad, bd, idesc, acc);
        }
        issued = true;
        commit(bar(BAR_EMPTY + s), C::ALL_CTAS);   // stage s free once these finish
        ++g;
      }
    }
    if (w.kb1 > w.kb0) {
      commit(bar(BAR_ACC_FULL + b), pair_mask);   // accumulator b complete in the pair
    } else {
      // K == 0: no MMA ran; signal the accumulator barriers directly.
      if constexpr (CG == 1)
        mbar_arrive(bar(BAR_ACC_FULL + b));
      else
        for (int r = 0; r < CG; ++r)
          mbar_arrive_cluster(mapa_shared(bar(BAR_ACC_FULL + b), rank + r));
    }
  }
done:
  if (issued) {
    // Every MMA this thread issued has finished once this arrives; TMEM can
    // then be freed even on the abort path.
    commit(bar(BAR_MMA_DRAIN), static_cast<uint16_t>(1u << rank));
    wait_drain(bar(BAR_MMA_DRAIN), 0);
  }
}

// ------------------------------------------------------------ epilogue

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Epilogue of a launch with wide D stores (short K, beta == 0, no stream-out,
// no split pieces): D leaves in 32 x 64 blocks (128-byte rows, 128-byte
// swizzle), half the TMA store rows of 32 x 32 blocks, which is what bounds a
// short-K GEMM's epilogue. Warp (q, hf) takes the unit's 64-column blocks jw
// with jw % 2 == hf through its own 4 KiB area of the epilogue region (laid
// out differently from the D slots, so a launch never mixes the two); one
// block in flight per warp. A loop of its own, apart from the general
// epilogue's: measured 2.7 % faster on 8192 x 8192 x 64 than the same steps
// as one branch of the general loop.
template <int CG>
__device__ __forceinline__ void epilogue_wide(const Params& p, uint32_t sbase, uint8_t* smem,
                                              uint32_t tmem_base, uint32_t rank, int warp,
                                              const Watchdog& wd) {
  using C = Cfg<CG>;
  const int lane = threadIdx.x & 31;
  const int e = warp - WARP_EPI0;
  const int q = warp & 3;
  const int hf = e / EPI_HALF_WARPS;
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8 * i; };
  const int cluster = blockIdx.x / C::CS, clusters = gridDim.x / C::CS;
  uint8_t* dq = smem + C::OFF_D + hf * (4 * WIDE_QUARTER_BYTES) + q * WIDE_QUARTER_BYTES;
  const uint32_t wrow = lane * 128, wswz = lane & 7;
  grid_dependency_wait();   // D may be read or written by the previous kernel
  int i = 0;
  Unit w;
  for (; next_unit(p, cluster, clusters, i, w); ++i) {
    const int l = w.l;
    const int row_tile = w.mb * C::CS + static_cast<int>(rank);
    const int m0 = row_tile * BM + 32 * q, n0 = w.n0;
    const int nwide = subtiles_in_part(p, row_tile, w) / 2;   // 64-column blocks: 0, 1, 2 or 4
    const uint32_t b = i & 1, aph = (i >> 1) & 1;
    const bool has_acc = w.kb1 > w.kb0;
    auto release_acc = [&]() {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (CG == 1 || rank % CG == 0)
          mbar_arrive(bar(BAR_ACC_EMPTY + b));
        else
          mbar_arrive_cluster(mapa_shared(bar(BAR_ACC_EMPTY + b), rank - rank % CG));
      }
    };
    if (!warp_wait_spin(bar(BAR_ACC_FULL + b), aph, wd)) break;
    tc_fence_after_sync();
#ifdef GEMM_WS_DEBUG
    if (p.trace && q == (WARP_EPI0 & 3) && hf == 0 && lane == 0)
      p.trace[(static_cast<size_t>(w.id) * C::CS + rank) * 2] = global_timer_ns();
#endif
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN;
    if (hf >= nwide) release_acc();   // no block of this part for this warp
    for (int jw = hf; jw < nwide; jw += 2) {
      uint32_t a0[32], a1[32];
      if (has_acc) {
        tmem_ld_32x32b_x32(tacc + (2 * jw) * EPI_N, a0);
        tmem_ld_32x32b_x32(tacc + (2 * jw + 1) * EPI_N, a1);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) a0[x] = a1[x] = 0u;
      }
      if (jw + 2 >= nwide) release_acc();
      if (lane == 0) bulk_wait_read<0>();   // this warp's previous block has been read
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t* a = c < 4 ? a0 : a1;
        const int o = 8 * (c & 3);
        uint4 wv;
        wv.x = pack_bf16x2(p.alpha * __uint_as_float(a[o + 0]), p.alpha * __uint_as_float(a[o + 1]));
        wv.y = pack_bf16x2(p.alpha * __uint_as_float(a[o + 2]), p.alpha * __uint_as_float(a[o + 3]));
        wv.z = pack_bf16x2(p.alpha * __uint_as_float(a[o + 4]), p.alpha * __uint_as_float(a[o + 5]));
        wv.w = pack_bf16x2(p.alpha * __uint_as_float(a[o + 6]), p.alpha * __uint_as_float(a[o + 7]));
        *reinterpret_cast<uint4*>(dq + wrow + ((c ^ wswz) << 4)) = wv;
      }
      fence_proxy_async_smem();   // generic writes -> visible to the TMA (async proxy)
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&p.tmDw, smem_addr(dq), n0 + jw * 2 * EPI_N, m0, l);
        bulk_commit();
      }
    }
#ifdef GEMM_WS_DEBUG
    if (p.trace && q == (WARP_EPI0 & 3) && hf == 0 && lane == 0)
      p.trace[(static_cast<size_t>(w.id) * C::CS + rank) * 2 + 1] = global_timer_ns();
#endif
  }
  if (lane == 0) bulk_wait_read<0>();   // store tail: shared memory read before the CTA exits
  __syncwarp();
}

template <int CG>
__device__ __forceinline__ void epilogue_role(const Params& p, uint32_t sbase, uint8_t* smem,
                                              uint32_t tmem_base, uint32_t rank, int warp,
                                              const Watchdog& wd) {
  using C = Cfg<CG>;
  const int lane = threadIdx.x & 31;
  const int e = warp - WARP_EPI0;    // epilogue warp 0..7
  const int q = warp & 3;            // TMEM lane quarter it may access = CTA rows 32q..32q+31
  const int hf = e / EPI_HALF_WARPS; // it takes the unit's subtiles j with j % 2 == hf
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8 * i; };
  // 64-byte swizzle of a 32-row x 64-byte block: 16-byte chunk c of row r is
  // stored at chunk c ^ ((r >> 1) & 3); the same pattern TMA uses.
  const uint32_t row_off = lane * 64;
  const uint32_t swz = (lane >> 1) & 3;
  const int cluster = blockIdx.x / C::CS, clusters = gridDim.x / C::CS;
  // Each half of the epilogue warps has its own ring of D slots: one (C is
  // read, its buffers take the space) or two.
  const uint32_t per_half = (p.has_c ? EPI_SLOTS : EPI_SLOTS_NOC) / 2;
  const uint32_t cbuf = sbase + C::OFF_C + static_cast<uint32_t>(e) * EPI_QUARTER_BYTES;
  const uint32_t cbar = bar(BAR_C_FULL + e);
  uint32_t u = 0;        // subtiles stored by this warp (slot ring position)
  uint32_t cu = 0;       // C subtiles consumed by this warp
  uint32_t c_issued = 0; // C subtile loads issued by this warp
  grid_dependency_wait();   // C and D may be the previous kernel's output or input
  int i = 0;
  Unit w;
  for (; next_unit(p, cluster, clusters, i, w); ++i) {
    const int l = w.l;
    const int row_tile = w.mb * C::CS + static_cast<int>(rank);   // this CTA's 128-row slab
    const int m0 = row_tile * BM + 32 * q, n0 = w.n0;
    const int nsub = subtiles_in_part(p, row_tile, w);   // 0, 2, 4 or 8
    const uint32_t b = i & 1, aph = (i >> 1) & 1;
    const bool has_acc = w.kb1 > w.kb0;   // an MMA ran (K > 0)

    // One C buffer per warp: the load for a subtile is issued as soon as the
    // previous subtile's C has been read out of it.
    auto issue_c = [&](int j) {
      ++c_issued;
      __syncwarp();                 // every lane has read the buffer's previous contents
      if (lane == 0) {
        fence_proxy_async_smem();   // ... before the TMA (async proxy) overwrites it
        mbar_arrive_expect_tx(cbar, EPI_QUARTER_BYTES);
        tma_load_3d(cbuf, &p.tmC, cbar, n0 + j * EPI_N, m0, l);
      }
    };
    auto release_acc = [&]() {
      // Accumulator b fully read by this warp: hand it back to the MMA warp
      // (the even CTA of the pair).
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (CG == 1 || rank % CG == 0)
          mbar_arrive(bar(BAR_ACC_EMPTY + b));
        else
          mbar_arrive_cluster(mapa_shared(bar(BAR_ACC_EMPTY + b), rank - rank % CG));
      }
    };
    // alpha * acc (+ beta * C) of subtile j, rounded to bf16, through a
    // shared-memory slot to the TMA store of D (and, with stream-out, to the
    // consumer warp). next_c: the subtile whose C load may now reuse this
    // warp's C buffer (-1: none). Returns false if a bounded wait gave up.
    auto finish_subtile = [&](int j, float (&v)[32], int next_c) -> bool {
      if (p.has_c) {
        if (!warp_wait_spin(cbar, cu & 1, wd)) return false;
        const uint8_t* cq = smem + (cbuf - sbase) + row_off;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 raw = *reinterpret_cast<const uint4*>(cq + ((c ^ swz) << 4));
          float cf[8];
          unpack_bf16x8(raw, cf);
#pragma unroll
          for (int x = 0; x < 8; ++x) v[8 * c + x] = fmaf(p.beta, cf[x], v[8 * c + x]);
        }
        ++cu;
        if (next_c >= 0) issue_c(next_c);
      }
      // Reuse a slot only when (a) this warp's TMA store from it has
      // finished reading it and (b) the stream-out consumer released it.
      const uint32_t slot = hf + 2 * (u % per_half);
      if (lane == 0) {
        if (per_half == 2)
          bulk_wait_read<1>();
        else
          bulk_wait_read<0>();
      }
      if (p.streamout) {
        if (!warp_wait_spin(bar(BAR_D_EMPTY + slot), ((u / per_half) & 1) ^ 1, wd)) return false;
      }
      __syncwarp();
      uint8_t* dq = smem + C::OFF_D + slot * EPI_SLOT_BYTES + q * EPI_QUARTER_BYTES;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 wv;
        wv.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
        wv.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
        wv.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
        wv.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(dq + row_off + ((c ^ swz) << 4)) = wv;
      }
      fence_proxy_async_smem();   // generic writes -> visible to the TMA (async proxy)
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&p.tmD, smem_addr(dq), n0 + j * EPI_N, m0, l);
        bulk_commit();
        if (p.streamout) mbar_arrive(bar(BAR_D_FULL + slot));
      }
      ++u;
      return true;
    };

    const bool split = w.pieces > 1;
    if (p.has_c && nsub > 0 && !split) issue_c(hf);

    if (!warp_wait_spin(bar(BAR_ACC_FULL + b), aph, wd)) break;
    tc_fence_after_sync();
#ifdef GEMM_WS_DEBUG
    // stamp 0: this CTA's part of the unit has its accumulator (MMA done)
    if (p.trace && q == (WARP_EPI0 & 3) && hf == 0 && lane == 0)
      p.trace[(static_cast<size_t>(w.id) * C::CS + rank) * 2] = global_timer_ns();
#endif
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN;

    // In-kernel fix-up of a two-piece tile: for this warp's chunks, the piece
    // whose warp arrives second adds the other piece's partial and runs the
    // epilogue; the first one writes its partial and flags it. The second
    // only ever waits for a piece that has already arrived (which writes
    // without waiting for anything), so no two clusters need to be resident
    // at once.
    bool reduce = false;
    if (split && p.sk_inline && hf < nsub) {
      uint32_t before = 0;
      if (lane == 0) before = atomicAdd(sk_arrival_word(p, C::CS, w.sk_tile, rank, e), 1u);
      before = __shfl_sync(0xffffffffu, before, 0);
      reduce = before == static_cast<uint32_t>(w.pieces - 1);
#ifdef GEMM_WS_DEBUG
      if (p.phases && e == 0 && lane == 0 && reduce) p.phases[blockIdx.x * 8 + 4] = global_timer_ns();
#endif
    }
    // The other piece's fp32 partial of this warp's chunks (reducer only),
    // bulk-copied into this warp's share of the ring's shared memory, which
    // the piece (its cluster's last unit) no longer loads into.
    const int nchunk = hf < nsub ? min(4, (nsub - hf + 1) / 2) : 0;
    const uint8_t* other = nullptr;
    uint8_t* fixbuf = smem + C::OFF_A + e * (4 * CHUNK_BYTES);
    if (reduce) {
      const int op = 1 - w.piece;
      if (p.has_c) issue_c(hf);
      uint32_t* written = sk_written_word(p, C::CS, sk_slot(p, w, op), rank, e);
      if (!warp_wait_flag(written, wd)) break;
#ifdef GEMM_WS_DEBUG
      if (p.phases && e == 0 && lane == 0) p.phases[blockIdx.x * 8 + 5] = global_timer_ns();
#endif
      if (lane == 0) {
        // Both pieces have arrived and the other is done with its flag: the
        // words go back to zero for the next launch.
        *sk_arrival_word(p, C::CS, w.sk_tile, rank, e) = 0u;
        *written = 0u;
        fence_proxy_async_global();   // the flag's acquire, then the bulk (async-proxy) read
        const float* src = p.partial +
                           (static_cast<size_t>(sk_slot(p, w, op)) * C::CS + rank) * PART_FLOATS +
                           part_chunk_offset(q, hf);
        // One copy (and barrier) per chunk, so the first subtile's sum can
        // start while the later chunks are still on their way.
        for (int k = 0; k < nchunk; ++k) {
          mbar_arrive_expect_tx(bar(BAR_FIX + 4 * e + k), CHUNK_BYTES);
          bulk_load_1d(smem_addr(fixbuf + k * CHUNK_BYTES), src + k * CHUNK_FLOATS, CHUNK_BYTES,
                       bar(BAR_FIX + 4 * e + k));
        }
      }
      other = fixbuf;
    }

    bool ok = true;
    if (!split || reduce) {
      if (nsub == 0) release_acc();   // this CTA's rows lie outside M x N
      for (int j = hf; j < nsub; j += 2) {
        uint32_t acc[32];
        if (has_acc) {
          tmem_ld_32x32b_x32(tacc + j * EPI_N, acc);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) acc[x] = 0u;
        }
        if (j + 2 >= nsub) release_acc();
        float v[32];
        if (other) {
          // The two partials in piece order, from zero: the same sum, bit
          // for bit, as the separate reduction kernel's.
          const bool first = w.piece == 0;
          if (!warp_wait_spin(bar(BAR_FIX + 4 * e + (j >> 1)), 0, wd)) {
            // The copies land before the CTA exits.
            if (lane == 0)
              for (int k = j >> 1; k < nchunk; ++k) wait_drain(bar(BAR_FIX + 4 * e + k), 0);
            ok = false;
            break;
          }
          const float4* oc = reinterpret_cast<const float4*>(other + (j >> 1) * CHUNK_BYTES) + lane;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 o = oc[c * 32];
            const float o4[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float mine = __uint_as_float(acc[4 * c + x]);
              const float s0 = first ? mine : o4[x], s1 = first ? o4[x] : mine;
              v[4 * c + x] = p.alpha * ((0.0f + s0) + s1);
            }
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = p.alpha * __uint_as_float(acc[x]);
        }
        if (!finish_subtile(j, v, j + 2 < nsub ? j + 2 : -1)) {
          ok = false;
          break;
        }
      }
    } else {
      // A piece of the tile's K range (every piece of a tile runs on its own
      // cluster, as that cluster's last unit): this warp's fp32 partial of
      // its 32 x 32 chunks (TMEM lane quarter q, subtiles j = hf + 2k) goes
      // to the piece's workspace part, each chunk in TMEM register order
      // (float4 c of lane r at [c][r]), the warp's chunks together
      // (part_chunk_offset). It passes through this warp's share of the
      // ring's shared memory (no more loads land there: the piece is its
      // cluster's last unit) and leaves in one bulk copy. Nothing here waits
      // for another piece. The partial is added either by the other piece's
      // warp (in-kernel fix-up, which this warp signals through its written
      // flag) or by the reduction kernel that follows on the stream (the
      // separate-reduction variant of the SM90 cooperative kernel's fix-up).
      for (int k = 0; k < nchunk; ++k) {
        uint32_t acc[32];
        tmem_ld_32x32b_x32(tacc + (hf + 2 * k) * EPI_N, acc);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(fixbuf + k * CHUNK_BYTES) + lane;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c * 32] = make_float4(__uint_as_float(acc[4 * c]), __uint_as_float(acc[4 * c + 1]),
                                    __uint_as_float(acc[4 * c + 2]), __uint_as_float(acc[4 * c + 3]));
      }
      release_acc();
#ifdef GEMM_WS_DEBUG
      if (p.phases && e == 0 && lane == 0) p.phases[blockIdx.x * 8 + 3] = global_timer_ns();
#endif
      if (nchunk > 0) {
        fence_proxy_async_smem();   // generic shared-memory writes -> the bulk copy
        __syncwarp();
        if (lane == 0) {
          float* part = p.partial +
                        (static_cast<size_t>(sk_slot(p, w, w.piece)) * C::CS + rank) * PART_FLOATS +
                        part_chunk_offset(q, hf);
          bulk_store_1d(part, smem_addr(fixbuf), nchunk * CHUNK_BYTES);
          bulk_commit();
          if (p.sk_inline) {
            // The partial is in global memory, then the flag (release, gpu
            // scope); the reduction kernel instead runs after this grid.
            bulk_wait<0>();
            fence_proxy_async_global();
#ifdef GEMM_WS_DEBUG
            if (p.debug_fault != 2)   // injected fault: the other piece waits in vain
#endif
            st_release_gpu(sk_written_word(p, C::CS, sk_slot(p, w, w.piece), rank, e), 1u);
#ifdef GEMM_WS_DEBUG
            if (p.phases && e == 0) p.phases[blockIdx.x * 8 + 6] = global_timer_ns();
#endif
          }
        }
      }
    }
    if (!ok) break;
#ifdef GEMM_WS_DEBUG
    // stamp 1 without stream-out: this warp issued the part's last D store
    if (p.trace && !p.streamout && q == (WARP_EPI0 & 3) && hf == 0 && lane == 0)
      p.trace[(static_cast<size_t>(w.id) * C::CS + rank) * 2 + 1] = global_timer_ns();
#endif
  }
  if (lane == 0) {
    // A C load still in flight only after an abort: let it land first.
    for (uint32_t idx = cu; idx < c_issued; ++idx) wait_drain(cbar, idx & 1);
    // Store tail: the D stores have finished reading shared memory, which
    // the CTA may release once every role is done. Their global writes are
    // performed before the grid completes, so nothing waits for them here.
    bulk_wait_read<0>();
  }
  __syncwarp();
}

// ------------------------------------------------------------ stream-out consumer

template <int CG>
__device__ __forceinline__ void consumer_role(const Params& p, uint32_t sbase, uint32_t rank,
                                              const Watchdog& wd) {
  using C = Cfg<CG>;
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8 * i; };
  const int cluster = blockIdx.x / C::CS, clusters = gridDim.x / C::CS;
  grid_dependency_wait();   // staging and flags may be in use by the previous kernel
  // Each stream-out tile has exactly one publishing consumer, which clears
  // the tile's flag words before anything else; so no host-side clearing is
  // needed and nothing in this launch can observe a stale ready word.
  Unit w;
  for (int it = 0; next_unit(p, cluster, clusters, it, w); ++it) {
    const int row_tile = w.mb * C::CS + static_cast<int>(rank);
    const int nst = staging_in_part(p, row_tile, w);
    for (int st = 0; st < nst; ++st) {
      const int tile_id =
          (w.l * p.staging_tiles_m + row_tile) * p.staging_tiles_n + w.n0 / STAGING + st;
      st_relaxed_gpu(p.flags + 2 * tile_id, 0u);
      st_relaxed_gpu(p.flags + 2 * tile_id + 1, 0u);
    }
  }
  // Subtile j of a unit sits in the ring of epilogue half j % 2.
  const uint32_t per_half = (p.has_c ? EPI_SLOTS : EPI_SLOTS_NOC) / 2;
  uint32_t uh[2] = {0, 0};   // subtiles taken from each half's ring
#ifdef GEMM_WS_DEBUG
  if (p.debug_fault == 1) goto done;   // injected fault: no tile is ever taken
#endif
  for (int it = 0; next_unit(p, cluster, clusters, it, w); ++it) {
    const int row_tile = w.mb * C::CS + static_cast<int>(rank);
    const int nst = staging_in_part(p, row_tile, w);
    for (int st = 0; st < nst; ++st) {
      const int tile_id =
          (w.l * p.staging_tiles_m + row_tile) * p.staging_tiles_n + w.n0 / STAGING + st;
      uint32_t seq = 0;
      for (int jj = 0; jj < SUB_PER_STAGING; ++jj) {
        const int hf = jj & 1;   // SUB_PER_STAGING is even: j % 2 == jj % 2
        const uint32_t k = uh[hf]++;
        const uint32_t slot = hf + 2 * (k % per_half);
        if (!wait_spin<false>(bar(BAR_D_FULL + slot), (k / per_half) & 1, wd)) goto done;
        if (jj == 0) seq = atomicAdd(p.counter, 1u);   // completion order
        tma_store_3d(&p.tmS, sbase + C::OFF_D + slot * EPI_SLOT_BYTES, jj * EPI_N, 0,
                     static_cast<int>(seq));
        bulk_commit();
        bulk_wait_read<0>();                  // slot read: give it back
        mbar_arrive(bar(BAR_D_EMPTY + slot));
      }
      bulk_wait<0>();                         // staging bytes written
      fence_proxy_async_global();
      __threadfence();
      st_relaxed_gpu(p.flags + 2 * tile_id, seq);
      st_release_gpu(p.flags + 2 * tile_id + 1, 1u);
    }
#ifdef GEMM_WS_DEBUG
    // stamp 1: every stream-out tile of this CTA's part of the unit is published
    if (p.trace && nst > 0)
      p.trace[(static_cast<size_t>(w.id) * C::CS + rank) * 2 + 1] = global_timer_ns();
#endif
  }
done:
  bulk_wait<0>();
  // The last consumer warp of the launch to get here (every one gets here,
  // also after an abort) zeroes the sequence counter for the next launch:
  // all counter updates of this launch happen before the arrivals on `done`.
  // So a call needs no host-side reset, and a launch replayed from a CUDA
  // graph starts from zero as well.
  __threadfence();
  if (atomicAdd(p.done, 1u) == gridDim.x - 1) {
    atomicExch(p.counter, 0u);
    atomicExch(p.done, 0u);
    __threadfence();
  }
}

// ------------------------------------------------------------ kernel

template <int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_ws_kernel(const __grid_constant__ Params p) {
  using C = Cfg<CG>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
  const int lane = threadIdx.x & 31;
  const uint32_t rank = C::CS == 1 ? 0u : cluster_ctarank();
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
#ifdef GEMM_WS_DEBUG
  unsigned long long t_entry = 0;
  if (p.phases && threadIdx.x == 0) t_entry = global_timer_ns();
#endif

  if (warp == WARP_TMA && lane == 0) {
    auto bar = [&](int i) { return sbase + C::OFF_BAR + 8 * i; };
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(BAR_FULL + s), 1);
      mbar_init(bar(BAR_EMPTY + s), 1);   // one MMA commit per stage
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(bar(BAR_ACC_FULL + b), 1);
      mbar_init(bar(BAR_ACC_EMPTY + b), NUM_EPI_WARPS * CG);
    }
    for (int i = 0; i < NUM_EPI_WARPS; ++i) mbar_init(bar(BAR_C_FULL + i), 1);
    for (int s = 0; s < EPI_SLOTS_NOC; ++s) {
      mbar_init(bar(BAR_D_FULL + s), EPI_HALF_WARPS);   // the four warps of one half
      mbar_init(bar(BAR_D_EMPTY + s), 1);
    }
    mbar_init(bar(BAR_MMA_DRAIN), 1);
    for (int i = 0; i < NUM_EPI_WARPS * 4; ++i) mbar_init(bar(BAR_FIX + i), 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (p.num_kb > 0) {
      prefetch_tensormap(&p.tmA);
      prefetch_tensormap(&p.tmB);
      if (p.num_full < p.num_tiles) prefetch_tensormap(p.split == 4 ? &p.tmB4 : &p.tmB2);
    }
    if (p.has_c) prefetch_tensormap(&p.tmC);
    prefetch_tensormap(&p.tmD);
    if (p.wide_d) prefetch_tensormap(&p.tmDw);
    if (p.streamout) prefetch_tensormap(&p.tmS);
  }
  if (warp == WARP_MMA) {
    if constexpr (CG == 1) {
      tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::CS > 1) cluster_sync();   // peers' barriers initialised before remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  // Everything above touches only this CTA's shared and tensor memory, so it
  // may overlap the previous kernel's tail. Global memory is touched only
  // after that kernel has completed: each role that reads or writes global
  // memory waits for it (grid_dependency_wait) just before its first such
  // access, so the rest of its set-up (unit coordinates, first barrier
  // waits, the first run of its code) overlaps the previous kernel too. The
  // MMA thread never touches global memory. The next launch may be
  // scheduled now (its CTAs take SMs as this grid's CTAs leave them).
  if (threadIdx.x == 0) grid_launch_dependents();
#ifdef GEMM_WS_DEBUG
  // Stamps per CTA: entry, start of work (after the previous grid; taken by
  // the A producer before its first copy), exit.
  if (p.phases && threadIdx.x == 0) p.phases[blockIdx.x * 8] = t_entry;
#endif

  if (warp == WARP_TMA || warp == WARP_TMA_B) {
    if (lane == 0)
      producer_role<CG>(p, sbase, rank, warp == WARP_TMA ? LOAD_A : LOAD_B, wd);
  } else if (warp == WARP_MMA) {
    if (lane == 0 && rank % CG == 0) mma_role<CG>(p, sbase, tmem_base, rank, wd);
  } else if (warp < WARP_EPI0 + NUM_EPI_WARPS) {
    if (p.wide_d)
      epilogue_wide<CG>(p, sbase, smem, tmem_base, rank, warp, wd);
    else
      epilogue_role<CG>(p, sbase, smem, tmem_base, rank, warp, wd);
  } else if (warp == WARP_CONSUMER && p.streamout) {
    if (lane == 0) consumer_role<CG>(p, sbase, rank, wd);
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  // The peer may still arrive on, or have the tensor core read, this CTA's
  // shared memory until both CTAs are here.
  if constexpr (C::CS > 1) cluster_sync();
  if (warp == WARP_MMA) {
    tc_fence_after_sync();
    if constexpr (CG == 1)
      tmem_dealloc(tmem_base, TMEM_COLS);
    else
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
#ifdef GEMM_WS_DEBUG
  if (p.phases && threadIdx.x == 0) p.phases[blockIdx.x * 8 + 2] = global_timer_ns();
#endif
}

// ------------------------------------------------------------ split reduction

// The pieces of the split tiles, combined: for every 32 x 32 chunk of a
// split tile's CTA part, the chunk's fp32 partials of all S pieces are added
// in piece order, then alpha * sum + beta * C is rounded to bf16 and stored
// to D. It runs as its own kernel after the GEMM on the same stream (the
// separate-reduction variant of the SM90 cooperative kernel's fix-up), so no
// piece ever waits for another and the GEMM needs no co-resident clusters.
struct ReduceParams {
  const float* partial;   // the GEMM's piece partials (see Params::partial)
  const uint16_t* C;      // L x M x N bf16, read iff has_c (may be D itself)
  uint16_t* D;            // L x M x N bf16
  int M, N;
  int tiles_m, tiles_n, group_m;   // the GEMM launch's tile grid and raster
  int cs;                          // CTAs per cluster: a tile has 128 * cs rows
  int sk_first, sk_tiles, sk_split;
  float alpha, beta;
  int has_c;
};

constexpr int REDUCE_THREADS = 256;   // one thread per float4 of a 32 x 32 chunk
constexpr int REDUCE_INFLIGHT = 8;    // pieces whose loads a thread keeps in flight

// One block per chunk. Thread t holds float4 c = t / 32 of chunk row r = t %
// 32 (the workspace layout, so the 256 threads read 4 KiB contiguously per
// piece), loads REDUCE_INFLIGHT pieces at a time and adds them in piece
// order; the sums then pass through shared memory so that C and D are read
// and written along rows.
__global__ void __launch_bounds__(REDUCE_THREADS)
    gemm_ws_reduce_kernel(const __grid_constant__ ReduceParams p) {
  __shared__ float sum[32][EPI_N + 4];   // padded rows: conflict-free both ways
  // The GEMM grid before this one in the stream has written every partial.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int x = blockIdx.x;                          // chunk
  const int per_part = 4 * SUB_PER_PART;             // chunks of one CTA's 128 x 256 part
  const int per_tile = p.cs * per_part;
  const int r = x / per_tile;
  const int rank = (x - r * per_tile) / per_part;
  const int cq = x - r * per_tile - rank * per_part;
  const int q = cq / SUB_PER_PART, j = cq - q * SUB_PER_PART;
  int mb, nb, l;
  tile_coords_of(p.tiles_m, p.tiles_n, p.group_m, p.sk_first + r, mb, nb, l);
  const int row_tile = mb * p.cs + rank;
  const int col0 = nb * BN + j * EPI_N;
  // Chunks outside M x N were not written by the pieces and hold no output.
  if (row_tile * BM >= p.M || col0 >= p.N) return;   // block-uniform
  const int t = threadIdx.x;
  const float4* src = reinterpret_cast<const float4*>(
                          p.partial + (static_cast<size_t>(r) * p.sk_split * p.cs + rank) *
                                          PART_FLOATS +
                          part_chunk_offset(q, j)) +
                      t;
  const size_t piece_stride = static_cast<size_t>(p.cs) * PART_FLOATS / 4;   // float4s
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int s0 = 0; s0 < p.sk_split; s0 += REDUCE_INFLIGHT) {
    float4 f[REDUCE_INFLIGHT];
#pragma unroll
    for (int k = 0; k < REDUCE_INFLIGHT; ++k)
      if (s0 + k < p.sk_split) f[k] = __ldcg(src + (s0 + k) * piece_stride);
#pragma unroll
    for (int k = 0; k < REDUCE_INFLIGHT; ++k) {
      if (s0 + k < p.sk_split) {
        acc.x += f[k].x;
        acc.y += f[k].y;
        acc.z += f[k].z;
        acc.w += f[k].w;
      }
    }
  }
  {
    const int cr = t % 32, c4 = t / 32;   // chunk row, float4 column
    sum[cr][4 * c4] = acc.x;
    sum[cr][4 * c4 + 1] = acc.y;
    sum[cr][4 * c4 + 2] = acc.z;
    sum[cr][4 * c4 + 3] = acc.w;
  }
  __syncthreads();
  // Row-wise epilogue: thread t takes 4 columns of chunk row t / 8.
  const int cr = t / 8, c0 = 4 * (t % 8);
  const int row = row_tile * BM + 32 * q + cr;
  if (row >= p.M || col0 + c0 >= p.N) return;        // N is a multiple of 8
  const size_t at = (static_cast<size_t>(l) * p.M + row) * p.N + col0 + c0;
  float o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = sum[cr][c0 + k] * p.alpha;
  if (p.has_c) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p.C + at);
    o[0] = fmaf(p.beta, __uint_as_float(raw.x << 16), o[0]);
    o[1] = fmaf(p.beta, __uint_as_float(raw.x & 0xFFFF0000u), o[1]);
    o[2] = fmaf(p.beta, __uint_as_float(raw.y << 16), o[2]);
    o[3] = fmaf(p.beta, __uint_as_float(raw.y & 0xFFFF0000u), o[3]);
  }
  uint2 out;
  out.x = pack_bf16x2(o[0], o[1]);
  out.y = pack_bf16x2(o[2], o[3]);
  *reinterpret_cast<uint2*>(p.D + at) = out;
}

}  // namespace gws

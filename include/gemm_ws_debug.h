/*
 * gemm_ws_debug.h — test hooks of the debug build of the GEMM library
 * (libgemm_ws_debug.so, compiled with -DGEMM_WS_DEBUG). The production
 * library (libgemm_ws.so) does not export these functions.
 *
 * The hooks serve two checks:
 *  - the watchdog: a run whose stream-out consumer warp never takes a tile
 *    must end on its own, report GEMM_WS_ERR_TIMEOUT through
 *    gemm_ws_query_status (or, for the allocation-free entry point, leave
 *    every ready word at 0), and leave the device usable;
 *  - overlap of the tile handoff with compute, the property the issue
 *    "How to build a pipeline between epilogue and communication warp
 *    groups?" asks to be shown: per-tile global-timer stamps of "accumulator
 *    complete" and "tile published".
 */
#ifndef GEMM_WS_DEBUG_H_
#define GEMM_WS_DEBUG_H_

#include <stdint.h>

#include "gemm_ws.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Sets the handle's debug state for its later runs.
 *  - fault: 0 none; 1 the stream-out consumer warp returns at once, so the
 *    epilogue's wait for a free slot can only end by the watchdog; 2 split
 *    pieces that write their partial for the in-kernel fix-up never set
 *    their written flag, so the piece that adds it can only stop waiting by
 *    the watchdog (its fix-up words are then left part-way, for
 *    gemm_ws_query_status to clear).
 *  - trace: device buffer of num_units * ctas_per_cluster * 2 uint64 (see
 *    gemm_ws_debug_launch_shape) or NULL. For work unit u and CTA rank r
 *    in its cluster, trace[(u*ctas_per_cluster + r)*2] = global time (ns) at which
 *    that CTA's epilogue saw the unit's accumulator complete, and [...+1] =
 *    with gemm_ws_run_streamout, time at which its consumer published the
 *    last stream-out tile of that part (untouched where the part lies
 *    outside M x N); with gemm_ws_run, time at which one epilogue warp (of
 *    the first lane quarter's even subtiles) issued its last D store of the
 *    unit. The caller owns the buffer.
 * Returns GEMM_WS_OK or GEMM_WS_ERR_INVALID_ARG. */
int gemm_ws_debug_configure(gemm_ws_t* h, int fault, unsigned long long* trace);

/* Sets (or, with NULL, clears) a device buffer of 8 uint64 per CTA of the
 * handle's later launches (size it with gemm_ws_debug_launch_shape:
 * clusters * ctas_per_cluster CTAs): for CTA b, phases[8b] = global time
 * (ns) at kernel entry, [8b+1] = after the wait for the previous grid in
 * the stream, [8b+2] = at exit; for the CTA's split piece, as seen by its
 * first epilogue warp: [8b+3] its partials written to the workspace. Slots
 * not reached stay as the caller left them. The
 * caller owns the buffer. Returns GEMM_WS_OK or GEMM_WS_ERR_INVALID_ARG. */
int gemm_ws_debug_phases(gemm_ws_t* h, unsigned long long* phases);

/* The launch the handle would make for an M x N x K x L problem (streamout:
 * nonzero for gemm_ws_run_streamout, 0 for gemm_ws_run): CTAs per cluster
 * (1 or 2), number of clusters (persistent CTA groups),
 * an upper bound of the work-unit ids (size the trace buffer with it), the
 * number of tiles in the stream-K region (0: every tile runs whole or in
 * parts), and, where the last two pointers are not NULL, the pieces per
 * split tile (1: none) and whether the GEMM kernel itself adds them (1) or
 * the reduction kernel does (0). Host arithmetic only.
 * Returns GEMM_WS_OK or GEMM_WS_ERR_INVALID_ARG (null output pointer, M, N or
 * L below 1, K below 0). */
int gemm_ws_debug_launch_shape(gemm_ws_t* h, int64_t M, int64_t N, int64_t K, int64_t L,
                               int streamout, int* ctas_per_cluster, int* clusters,
                               int* num_units, int* sk_tiles, int* sk_pieces, int* sk_inline);

/* The whole persistent schedule of a launch, on the host, without a handle
 * or a GPU: the plan the library makes for a device with `num_sms` SMs on
 * which `max_clusters` clusters of the chosen shape fit (cta_group 1 or 2,
 * or 0 to let the library choose per problem with `max_clusters` CTA pairs
 * and `num_sms` single CTAs; stream_k 0 off / 1 cost
 * model / 2 always), and the units
 * every cluster walks, produced by the kernel's own unit iterator.
 *  - plan[9] = {CTAs per cluster, clusters, unit-id bound, tiles, ring
 *    stages per tile, first stream-K tile, stream-K clusters, tiles_m,
 *    tiles_n}.
 *  - rows: NULL, or max_rows x 15 ints, one row per unit in cluster-then-
 *    walk order: {cluster, i, id, tile, m block, first column, width,
 *    batch, first stage, end stage, piece, pieces, stream-K tile, cluster of
 *    piece 0, workspace slot (-1 for a whole tile)}; *num_rows = units.
 * Returns GEMM_WS_OK or GEMM_WS_ERR_INVALID_ARG. */
int gemm_ws_debug_schedule(int cta_group, int num_sms, int max_clusters, int stream_k,
                           int64_t M, int64_t N, int64_t K, int64_t L, int streamout, int* rows,
                           int64_t max_rows, int64_t* num_rows, int* plan);

/* Debug state of gemm_ws_run_streamout_noalloc on CUDA device `device`, for
 * its later calls in this process: fault 0 none, 1 the stream-out consumer
 * warp takes no tile (as fault 1 of gemm_ws_debug_configure), so the run
 * can only end by the watchdog; timeout_ms > 0 replaces the per-wait limit,
 * 0 restores the default. Returns GEMM_WS_OK or GEMM_WS_ERR_INVALID_ARG. */
int gemm_ws_debug_noalloc_configure(int device, int fault, long long timeout_ms);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_WS_DEBUG_H_ */

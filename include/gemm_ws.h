/*
 * gemm_ws.h — C ABI of the GB300 (sm_103a) persistent warp-specialized GEMM
 *
 *   D[l] = alpha * A[l] * B[l] + beta * C[l]      for l = 0 .. L-1
 *
 * bf16 operands, fp32 accumulation in tensor memory, bf16 output.
 *
 * Where the operation is defined:
 *  - "sm90_gemm_tma_warpspecialized_cooperative.hpp" (CUTLASS kernel layer):
 *    the MNKL problem shape (rank-4 problem with an appended batch mode L),
 *    the host-side `can_implement` / workspace conventions, and the epilogue
 *    that reads C and writes D = alpha * accumulator + beta * C;
 *  - "How to build a pipeline between epilogue and communication warp
 *    groups?" (CUTLASS issue): the per-tile producer/consumer handoff from
 *    the epilogue to a separate consumer warp, which this library implements
 *    as the stream-out consumer (gemm_ws_run_streamout);
 *  - "why does load() pre-issue producer_try_acquire for the next stage"
 *    (CUTLASS discussion): the TMA producer's early try-acquire.
 *
 * Layouts (all packed, no padding between batches):
 *  - A: L x M x K row-major (K contiguous);
 *  - B: column-major K x N per batch, i.e. stored L x N x K with K contiguous;
 *  - C, D: L x M x N row-major.
 * Element type: IEEE bfloat16 bit patterns (uint16_t).
 *
 * Ownership: every data pointer is a borrowed DEVICE pointer on the handle's
 * device; the caller owns it and keeps it alive until the stream work ends.
 * The handle owns only its device workspace: the stream-out sequence
 * counter, a status word, a completion count, the split-K area (one
 * 128 x 256 fp32 partial per SM, 128 KiB per SM) and the split tiles'
 * arrival counts and written flags (64 bytes per SM).
 * The kernel returns every counter to zero before it ends, so runs need no
 * clearing between them; runs on one handle that overlap on the GPU (e.g. on
 * two streams) race on that workspace: serialise them or use one handle per
 * stream.
 *
 * Threads: a handle is not thread-safe (each call also updates its host-side
 * cache of TMA descriptors); calls on one handle from several host threads
 * must be serialised by the caller. Different handles are independent.
 * gemm_ws_run_streamout_noalloc takes a library-wide lock only for its
 * one-time per-device set-up.
 *
 * Errors: every entry point returns a gemm_ws_status. A call that returns an
 * error other than GEMM_WS_ERR_CUDA launched nothing and wrote nothing. All
 * runs are asynchronous on `stream` (a cudaStream_t passed as void*, NULL
 * meaning the legacy default stream); device-side problems (a watchdog
 * timeout) are reported by gemm_ws_query_status.
 */
#ifndef GEMM_WS_H_
#define GEMM_WS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_ws_status {
  GEMM_WS_OK = 0,
  GEMM_WS_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, beta != 0 with C NULL,
                                  D aliasing A or B, a size beyond the limits below */
  GEMM_WS_ERR_ALIGNMENT = 2,   /* a pointer not 16-byte aligned, or K or N not a
                                  multiple of 8 (TMA needs 16-byte row pitches) */
  GEMM_WS_ERR_UNSUPPORTED = 3, /* device is not sm_103 (GB300) */
  GEMM_WS_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed; see
                                  gemm_ws_last_cuda_error */
  GEMM_WS_ERR_TIMEOUT = 5      /* a bounded on-device wait gave up (watchdog) */
} gemm_ws_status;

typedef struct gemm_ws gemm_ws_t;

/* Creates a handle bound to CUDA device `device`: checks that it is sm_103,
 * queries its SM count, allocates the device workspace and sets the kernel's
 * shared-memory attribute. The caller owns *out and frees it with
 * gemm_ws_destroy. On error *out is set to NULL.
 * Defined by: "sm90_gemm_tma_warpspecialized_cooperative.hpp", the host
 * side of the kernel layer (`get_workspace_size` / `initialize_workspace`:
 * the scheduler's workspace is sized and set up once, before any launch;
 * here it lives as long as the handle). */
int gemm_ws_create(gemm_ws_t** out, int device);

/* Frees the handle and its workspace (synchronising the device first). NULL
 * is accepted and ignored.
 * Defined by: the same header's workspace convention (the caller releases
 * what initialize_workspace set up once no launch uses it). */
int gemm_ws_destroy(gemm_ws_t* h);

/* D[l] = alpha * A[l] * B[l] + beta * C[l], asynchronously on `stream`.
 *  - A: L*M*K, B: L*N*K, C: L*M*N (may be NULL iff beta == 0, in which case C
 *    is never read), D: L*M*N; all bf16, layouts as above.
 *  - M, N, K, L >= 0, each < 2^31, and L*M*N, L*M*K, L*N*K < 2^40.
 *  - K % 8 == 0 and N % 8 == 0 (16-byte row pitches); pointers 16-byte aligned.
 *  - K == 0 gives D = beta * C (or 0); M*N*L == 0 launches nothing.
 *  - D must not overlap A or B; D may be exactly C (in place).
 * Rounding: fp32 alpha * acc + beta * c, then round-to-nearest-even to bf16.
 * Split-K / stream-K pieces: when the output has at most half as many tiles
 * as the GPU has persistent clusters and K is long, or the last wave of
 * tiles is at most half full, those tiles' K ranges may be cut into 2..16
 * equal pieces of >= 1024 that run on separate clusters (chosen by a host
 * cost model); acc is then the sum, in piece order, of the pieces' fp32
 * partials (deterministic: the same bits on every run). With two pieces the
 * GEMM kernel adds them itself: per epilogue warp, the piece that arrives
 * second waits for the other's partial (written to the workspace and
 * flagged), adds it and writes D; it waits only for a piece that has already
 * arrived. With more pieces, every piece writes its partial and waits for
 * nothing; a second, small kernel that the call launches after the GEMM on
 * the same stream adds them and writes those tiles' D. Both give the same
 * bits, and neither needs the pieces to run at the same time, so the call
 * works on a GPU shared with other kernels too. GEMM_WS_SK_INLINE=0 in the
 * environment at gemm_ws_create sends two-piece tiles to the reduction
 * kernel as well.
 * GEMM_WS_STREAM_K in the environment at gemm_ws_create sets this per
 * handle: 0 off, 1 (default) by the cost model, 2 wherever the shape allows
 * (pieces down to one ring stage). gemm_ws_run_streamout never splits.
 * Other per-problem choices change only the fp32 summation order, which is
 * fixed for a given problem and handle (the same bits on every run): the
 * tile configuration (CTA pairs or single CTAs; GEMM_WS_CTA_GROUP=1|2 forces
 * one) and walking every other unit's K range backwards (GEMM_WS_K_SNAKE=0
 * turns that off).
 * Defined by: "sm90_gemm_tma_warpspecialized_cooperative.hpp": the rank-4
 * MNKL problem shape of `Arguments`, the `can_implement` checks, the
 * mainloop (producer warp group loading A and B stages, consumer warp groups
 * accumulating) and the epilogue of `operator()` (`collective_epilogue.load`
 * of C, `collective_epilogue.store` of alpha * accumulator + beta * C);
 * "why does load() pre-issue producer_try_acquire for the next stage": the
 * producer ring's early try-acquire. */
int gemm_ws_run(gemm_ws_t* h, const uint16_t* A, const uint16_t* B,
                const uint16_t* C, uint16_t* D, int64_t M, int64_t N, int64_t K,
                int64_t L, float alpha, float beta, void* stream);

/* gemm_ws_run plus tile stream-out: a consumer warp takes every finished
 * 128 x 128 output tile from the epilogue through an on-chip full/empty
 * handoff and copies it into `staging`, in the order it takes the tiles.
 *  - T = L * ceil(M/128) * ceil(N/128) output tiles; tile index
 *    t = (l * ceil(M/128) + m_tile) * ceil(N/128) + n_tile.
 *  - staging: device buffer of T * 128 * 128 bf16; slot s holds, row-major
 *    128 x 128, the tile that was taken s-th; elements of an edge tile outside
 *    M or N are 0.
 *  - flags: device buffer of 2 * T uint32. After the stream work completes,
 *    flags[2t] = s (the slot / sequence number of tile t, 0-based and dense)
 *    and flags[2t+1] = 1. Within the launch, the warp that publishes a tile
 *    first clears that tile's two words, then writes the ready word with
 *    release semantics after the tile's staging bytes are globally visible.
 *    (No host-side memset: the call launches exactly one kernel.)
 *  - staging and flags must not overlap any other argument.
 * Returns as gemm_ws_run.
 * Defined by: "How to build a pipeline between epilogue and communication
 * warp groups?" (CUTLASS issue): the epilogue, as producer, acquires a
 * buffer, stores a finished tile and commits it; a separate consumer warp
 * waits for it, does its work on the tile and releases the buffer, while the
 * MMA warps go on with the next tile. The issue's closing request, to show
 * overlap and a correct handoff, is what the staging copy, sequence numbers
 * and ready words make checkable. */
int gemm_ws_run_streamout(gemm_ws_t* h, const uint16_t* A, const uint16_t* B,
                          const uint16_t* C, uint16_t* D, int64_t M, int64_t N,
                          int64_t K, int64_t L, float alpha, float beta,
                          uint16_t* staging, uint32_t* flags, void* stream);

/* Synchronises `stream` and returns the device status word of the handle:
 * GEMM_WS_OK, or GEMM_WS_ERR_TIMEOUT if a run's bounded wait gave up (the
 * run's outputs are then undefined). Reading a non-zero word clears it and
 * returns the workspace counters to zero; after a timeout, call this before
 * the next run on the handle.
 * Defined by: no page; every wait in the kernel is bounded (the cited
 * kernels' waits are not), and this call reads the result of those bounds. */
int gemm_ws_query_status(gemm_ws_t* h, void* stream);

/* The last CUDA error code (cudaError_t value) seen by this handle, 0 if none. */
int gemm_ws_last_cuda_error(gemm_ws_t* h);

/* A static, human-readable name for a gemm_ws_status value. */
const char* gemm_ws_status_string(int status);

/* Output tiles (128 x 128) of an M x N x L problem: the T of
 * gemm_ws_run_streamout. Pure host arithmetic; needs no GPU. */
int64_t gemm_ws_streamout_tiles(int64_t M, int64_t N, int64_t L);

/* Kernels that a run of this problem on this handle launches on its stream:
 * 1, or 2 when some tiles are split into more than two K pieces (the GEMM,
 * then the reduction of the pieces); 0 for an empty problem (M*N*L == 0); negative
 * (a gemm_ws_status, negated) for invalid sizes or a NULL handle. streamout:
 * nonzero for gemm_ws_run_streamout, which never splits. Host arithmetic
 * only, the same plan the run makes; useful for counting launches or sizing
 * CUDA-graph captures.
 * Defined by: no page; the SM90 cooperative kernel header's separate-
 * reduction variant of the stream-K fix-up is what adds the second kernel. */
int gemm_ws_kernels_per_run(gemm_ws_t* h, int64_t M, int64_t N, int64_t K, int64_t L,
                            int streamout);

/* gemm_ws_run_streamout for callers that cannot allocate device memory.
 *
 * The cited CUTLASS sources have no counterpart: this is a library
 * convenience. Some callers
 * may not call cudaMalloc (code that runs inside another allocator's hook, a
 * framework that owns and pools every device allocation, a process that
 * reserved all device memory up front), so they cannot create the handle,
 * whose workspace is cudaMalloc'ed. This call needs no handle and allocates
 * nothing: it runs on the CURRENT device, and its scratch (the 32-bit
 * stream-out sequence counter and the watchdog status word) is a fixed
 * 256-byte array in the library's device memory, which every GPU that loads
 * the library holds until the process exits.
 *  - Arguments, layouts, results and errors are those of
 *    gemm_ws_run_streamout. A problem of more than 2^31 - 1 stream-out tiles
 *    (beyond what the scratch counter numbers) returns
 *    GEMM_WS_ERR_INVALID_ARG.
 *  - The first call on a device does a one-time set-up there (device
 *    checks, kernel attribute, address of the scratch array); make that first
 *    call before any stream capture.
 *  - Every call shares the one scratch array, which keeps the last call's
 *    contents. The kernel returns its sequence counter to zero before it
 *    ends, so consecutive calls need no clearing. Calls that overlap on the
 *    GPU (e.g. on two streams) race on the counter and produce wrong sequence
 *    numbers: serialise them.
 *  - A watchdog timeout is not reported through a status query here; it shows
 *    as tiles whose ready word flags[2t+1] stayed 0 (the kernel also records
 *    it in a scratch word that no call reads). The next call starts from a
 *    zero sequence counter all the same. */
int gemm_ws_run_streamout_noalloc(const uint16_t* A, const uint16_t* B,
                                  const uint16_t* C, uint16_t* D, int64_t M,
                                  int64_t N, int64_t K, int64_t L, float alpha,
                                  float beta, uint16_t* staging, uint32_t* flags,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_WS_H_ */

/*
 * libmxa2a — fused AllToAll + MXFP8 block-scaled GEMM for NVIDIA GB300 (sm_103a).
 *
 * The operation is the MC2 "AllToAll + quantised matmul" kernel of the
 * all_to_all_matmul example (all_to_all_matmul_impl.h, class
 * AllToAllQuantMatmulImpl: AllToAllProcess stages the R K-segments of A
 * through a ring of bufferSize slots of commMSize rows; MatmulProcess runs a
 * block-scaled FP8 GEMM over every staged slot with split-K over the R
 * segments and writes BF16).  On one GPU the R "ranks" are R separate device
 * buffers A_seg[0..R-1]; the library stages them through its own ring and
 * computes, for every m < M, n < N:
 *
 *   C[m][n] = bf16( sum_{r<R} sum_{k<kPerRank}
 *                    e4m3(A_seg[r][m][k])      * 2^(A_scale_seg[r][m][k/32] - 127)
 *                  * e4m3(B[n][r*kPerRank + k]) * 2^(B_scale[n][(r*kPerRank + k)/32] - 127) )
 *
 * accumulated in fp32 on the tensor cores and rounded once to BF16 (round to
 * nearest even).  K = R * kPerRank.
 *
 * Data types and layouts (all row-major, all device memory unless noted):
 *   A_seg[r]        uint8 E4M3 ("fn": no infinities, 0x7F/0xFF are NaN), [M][kPerRank]
 *   A_scale_seg[r]  uint8 E8M0 (2^(x-127), 0xFF = NaN), [M][kPerRank/32]
 *   B               uint8 E4M3, [N][K]  (B is logically K x N, stored transposed:
 *                   the kernel entry's TransB = true)
 *   B_scale         uint8 E8M0, [N][K/32]
 *   C_bf16          uint16 BF16 bit patterns, [M][N]
 * Alignment: A_seg[r], B and C_bf16 16-byte aligned; scale pointers 4-byte aligned.
 *
 * Ownership: the caller owns every input and output buffer and the stream;
 * the plan owns its device workspace (staging ring, scale-factor tiles, credit
 * counters, split-K partials, status block), allocated by mxa2a_create on the
 * current device and freed by mxa2a_destroy.  Runs are asynchronous on the
 * given stream; one plan must not run on two streams at once.
 *
 * Errors: every int-returning call returns MXA2A_OK (0) or an MXA2A_ERR_* code
 * and never aborts the process.  Device-side failures (a bounded wait that ran
 * out) are reported by mxa2a_get_status after the stream has been synchronised.
 */
#ifndef MXA2A_H
#define MXA2A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum mxa2a_error {
    MXA2A_OK = 0,
    MXA2A_ERR_INVALID_SHAPE = 1,      /* shape rule broken (see mxa2a_validate) */
    MXA2A_ERR_NULL_PTR = 2,           /* a required pointer is NULL */
    MXA2A_ERR_MISALIGNED = 3,         /* pointer alignment rule broken */
    MXA2A_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    MXA2A_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
    MXA2A_ERR_TIMEOUT = 6,            /* device: a bounded wait ran out (get_status) */
    MXA2A_ERR_INVALID_OPTION = 7,     /* unknown option key or value out of range */
    MXA2A_ERR_DEVICE_CHECK = 8,       /* device: an internal consistency check failed */
    MXA2A_ERR_WRONG_DEVICE = 9,       /* current device differs from the plan's */
    MXA2A_ERR_SCRATCH_TOO_SMALL = 10, /* mxa2a_run_noalloc: the problem needs more than its static scratch */
    MXA2A_ERR_CAPTURE_SPLIT = 11      /* a run with a K split was issued while its stream is being captured
                                         into a CUDA graph (not supported, see mxa2a_run) */
};

typedef struct mxa2a_plan mxa2a_plan;   /* opaque */

/* Device-side status of the runs since the previous mxa2a_get_status call. */
typedef struct mxa2a_status {
    int32_t code;       /* MXA2A_OK, or the first device error of the reported launch */
    int32_t role;       /* 1 staging copy, 2 TMA producer, 3 MMA issuer, 4 epilogue, 5 exit,
                           6 reduce-scatter sum */
    int32_t block;      /* CTA that reported */
    int32_t step;       /* staging step waited on, -1 if none */
    int32_t segment;    /* segment waited on, -1 if none */
    int32_t slot;       /* ring slot waited on, -1 if none */
    int64_t observed;   /* counter value seen when the wait gave up */
    int64_t expected;   /* value it waited for */
    int64_t launch;     /* index (1-based, per plan) of the launch that failed */
} mxa2a_status;

/*
 * Shape rules, checked by mxa2a_validate and mxa2a_create (the pages take
 * m, k, n and rankNum, require k % rankNum == 0 and CeilDiv(k/rankNum, 64)
 * even, and silently drop rows when commMSize does not divide m; here every
 * rule is an error instead):
 *   1 <= R <= 64; M >= 1; kPerRank % 128 == 0; N % 16 == 0, N >= 16;
 *   commMSize % 64 == 0; M % commMSize == 0; 1 <= buffer_num <= 8;
 *   buffer_num >= the number of staging steps one 128-row output tile spans
 *   (2 when commMSize is 64 or not a multiple of 128, else 1);
 *   M, N, K <= 2^20.
 * Returns MXA2A_OK or MXA2A_ERR_INVALID_SHAPE.  Pure host code.
 * Passage: all_to_all_matmul.cpp (the launcher), its argument checks (m, k, n,
 * rankNum positive; k divisible by rankNum; CeilDiv(Ka, 64) even) and the
 * [MODIFY C2] note that headMSize must divide m or the tail block is lost.
 */
int mxa2a_validate(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num);

/*
 * Create a plan for one problem shape on the current CUDA device: validates
 * the shape, derives the tiling (128x256 output tiles, 128-wide K blocks,
 * split-K over segments when there are too few tiles to fill the GPU),
 * allocates the workspace and encodes the TMA descriptors of the ring.
 * Arguments: R segments ("ranks"), M rows of A and C, kPerRank = K extent of
 * one segment, N columns of C, commMSize rows per staging step, buffer_num
 * ring slots.  The plan (and its device workspace) belongs to the caller
 * until mxa2a_destroy.  Returns NULL on error; mxa2a_last_error() then gives
 * the code (MXA2A_ERR_INVALID_SHAPE, MXA2A_ERR_UNSUPPORTED_DEVICE, or
 * MXA2A_ERR_CUDA when an allocation or a descriptor encoding failed).
 * Passage: all_to_all_matmul.cpp (the launcher), runAllToAllMatmul: the
 * tiling it fills before the launch (commTilingData.tileCnt from headMSize,
 * [MODIFY C2]; bufferSize, [MODIFY C1]; the tile GEMM tiling for headMSize x
 * n x Ka) and the communication space it reserves (rankSize * bufferSize *
 * bufferBlockSize + scales); here the plan holds both.
 */
mxa2a_plan *mxa2a_create(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num);

/* Error code of the last failed mxa2a_create* on this thread (MXA2A_OK after
 * a successful one).  Thread-local; no side effects.
 * Passage: all_to_all_matmul.cpp (the launcher), its ACL_CHECK wrapping of
 * every runtime call: a failed call is reported, here as a code the caller
 * reads instead of a message. */
int mxa2a_last_error(void);

/* What a plan computes (mxa2a_get_option(MXA2A_INFO_KIND)). */
enum mxa2a_kind {
    MXA2A_KIND_ALLTOALL = 0,       /* mxa2a_create: AllToAll + GEMM (above) */
    MXA2A_KIND_ALLGATHER = 1,      /* mxa2a_create_allgather: AllGather + GEMM */
    MXA2A_KIND_REDUCE_SCATTER = 2, /* mxa2a_create_reduce_scatter: GEMM + ReduceScatter */
    MXA2A_KIND_ALLREDUCE = 3       /* mxa2a_create_allreduce: GEMM + AllReduce (one-shot) */
};

/*
 * AllGather + GEMM, the first fused-operator case of the performance
 * optimisation guide (section 3.1, which gives the title only; this is the
 * plain reading of the name).  R ranks each hold a block of rowsPerRank rows
 * of A with all K columns; the all-gather stacks the blocks along M =
 * R * rowsPerRank, and the rank multiplies the gathered A by its own B:
 *
 *   C[j*rowsPerRank + i][n] = bf16( sum_{k<K} e4m3(A_blk[j][i][k]) * 2^(A_scale_blk[j][i][k/32] - 127)
 *                                            * e4m3(B[n][k])       * 2^(B_scale[n][k/32] - 127) )
 *
 * On one GPU the R blocks are R device buffers: A_blk[j] uint8 [rowsPerRank][K],
 * A_scale_blk[j] uint8 [rowsPerRank][K/32].  The plan runs through the
 * all-to-all plan's calls, which then take A_blk / A_scale_blk (R pointers
 * each) in place of A_seg / A_scale_seg:
 *   mxa2a_run          fused: the blocks travel commMSize rows at a time
 *                      through the buffer_num-slot ring with the same credit
 *                      protocol, and the GEMM consumes each step as it lands;
 *   mxa2a_run_unfused  gather into one [M][K] operand, then the GEMM;
 *   mxa2a_run_direct   the GEMM reads the blocks in place (rowsPerRank % 128
 *                      == 0, else MXA2A_ERR_INVALID_OPTION);
 *   mxa2a_run_host     the fused run from host buffers (R blocks).
 * (mxa2a_run_noalloc computes the all-to-all only.)
 * There is one K slice, so no K split.  B, B_scale, C, element formats,
 * alignment, ownership, options and errors as for the all-to-all plan.
 * Shape rules: 1 <= R <= 64, rowsPerRank % commMSize == 0, and the
 * all-to-all rules for (R = 1, M = R * rowsPerRank, kPerRank = K, N,
 * commMSize, buffer_num).  Returns MXA2A_OK or MXA2A_ERR_INVALID_SHAPE.
 */
int mxa2a_validate_allgather(int R, int64_t rowsPerRank, int64_t K, int64_t N, int64_t commMSize, int buffer_num);
mxa2a_plan *mxa2a_create_allgather(int R, int64_t rowsPerRank, int64_t K, int64_t N, int64_t commMSize,
                                   int buffer_num);

/*
 * GEMM + ReduceScatter, the second fused-operator case of the performance
 * optimisation guide (section 3.2, title only; plain reading).  R ranks hold
 * K-sharded operands; rank `rank` holds A uint8 [M][K] (+ A_scale [M][K/32])
 * and B uint8 [N][K] (+ B_scale [N][K/32]), computes its partial
 * P = bf16(A x B^T) ([M][N], the block-scaled product of the all-to-all plan
 * with one segment) and reduce-scatters it: row block j (Mr = M / R rows) of
 * every rank's partial goes to rank j, which sums them.  The partials travel
 * as BF16 (the operation's output type) and are summed in fp32 in rank order
 * and rounded once to BF16, the arithmetic of a BF16 GEMM followed by a BF16
 * reduce-scatter.  From this rank's side, on one GPU:
 *
 *   send[j][i][n] = P[j*Mr + i][n]                             j != rank
 *   out[i][n]     = bf16( sum_{j<R} v_j[i][n] )  (fp32, j = 0, 1, .., R-1)
 *                   v_rank = P[rank*Mr + i][n],  v_j = recv[j][i][n] (j != rank)
 *
 * recv[j] is what peer j sent this rank and send[j] what this rank sends peer
 * j: host arrays of R device pointers to uint16 BF16 [Mr][N] buffers (entry
 * `rank` unused, may be NULL); out uint16 BF16 [Mr][N].  Alignment: A, B,
 * out, recv[j], send[j] 16 bytes; scales 4.
 *   mxa2a_run_reduce_scatter          fused: one persistent GEMM (A and B
 *       read in place) whose epilogue routes every finished tile, a peer's
 *       rows to its send buffer and this rank's to out; the kernel's spare
 *       warps then sum out's rows with the received partials in place, while
 *       the GEMM goes on with the peers' blocks (this rank's block is
 *       computed first);
 *   mxa2a_run_reduce_scatter_unfused  the GEMM writes P into a plan-owned
 *       [M][N] buffer, then a reduce-scatter kernel copies the peers' blocks
 *       and sums this rank's.
 * Both give the same bits.  Shape rules: 1 <= R <= 64, 0 <= rank < R,
 * M % (64 * R) == 0, K % 128 == 0, N % 16 == 0, M, N, K <= 2^20.  Options as
 * for the other kinds (no K split).  Returns NULL on error
 * (mxa2a_last_error).
 */
int mxa2a_validate_reduce_scatter(int R, int rank, int64_t M, int64_t K, int64_t N);
mxa2a_plan *mxa2a_create_reduce_scatter(int R, int rank, int64_t M, int64_t K, int64_t N);
int mxa2a_run_reduce_scatter(mxa2a_plan *plan, const void *A, const void *A_scale, const void *B,
                             const void *B_scale, const void *const *recv, void *const *send, void *out_bf16,
                             void *stream);
int mxa2a_run_reduce_scatter_unfused(mxa2a_plan *plan, const void *A, const void *A_scale, const void *B,
                                     const void *B_scale, const void *const *recv, void *const *send,
                                     void *out_bf16, void *stream);

/*
 * GEMM + AllReduce, one-shot: the third fused-operator case of the
 * performance optimisation guide (section 3.3, title only; plain reading).
 * The operands are K-sharded as for the reduce-scatter, and every rank ends
 * with the whole sum.  One-shot means that each rank publishes its partial
 * and reads every peer's partial directly, with no ring of partial sums.
 * From rank `rank`'s side, on one GPU, for all m < M, n < N:
 *
 *   pub[m][n] = P[m][n] = bf16(A x B^T)[m][n]        (this rank's published partial)
 *   out[m][n] = bf16( sum_{j<R} v_j[m][n] )  (fp32, j = 0, 1, .., R-1)
 *               v_rank = P[m][n],  v_j = recv[j][m][n] (j != rank)
 *
 * recv[j] is peer j's published partial: a host array of R device pointers
 * to uint16 BF16 [M][N] (entry `rank` unused, may be NULL); pub and out are
 * uint16 BF16 [M][N].  Alignment: A, B, pub, out, recv[j] 16 bytes; scales 4.
 *   mxa2a_run_allreduce          fused: one persistent GEMM whose epilogue
 *       publishes each finished tile to pub; the kernel's spare warps sum
 *       each tile's rows with the peers' partials into out as soon as
 *       it is published, while the GEMM goes on;
 *   mxa2a_run_allreduce_unfused  the GEMM writes pub, then a reduce kernel
 *       writes out.
 * Both give the same bits.  Shape rules: 1 <= R <= 64, 0 <= rank < R,
 * M % 64 == 0, K % 128 == 0, N % 16 == 0, M, N, K <= 2^20.  Returns NULL on
 * error (mxa2a_last_error).
 */
int mxa2a_validate_allreduce(int R, int rank, int64_t M, int64_t K, int64_t N);
mxa2a_plan *mxa2a_create_allreduce(int R, int rank, int64_t M, int64_t K, int64_t N);
int mxa2a_run_allreduce(mxa2a_plan *plan, const void *A, const void *A_scale, const void *B, const void *B_scale,
                        const void *const *recv, void *pub_bf16, void *out_bf16, void *stream);
int mxa2a_run_allreduce_unfused(mxa2a_plan *plan, const void *A, const void *A_scale, const void *B,
                                const void *B_scale, const void *const *recv, void *pub_bf16, void *out_bf16,
                                void *stream);

/*
 * The fused path: one persistent cooperative kernel stages A_seg[r] rows
 * (commMSize per step, buffer_num-slot ring, per-segment credits) and runs
 * the block-scaled GEMM on the staged slots as they fill; its prologue
 * reorders B_scale for the MMA.  When the ring holds too few output tiles to
 * fill the GPU, K is split over segment groups and the split partials are
 * summed inside the kernel in a fixed order (deterministic).
 * A_seg / A_scale_seg are host arrays of R device pointers.  stream is a
 * cudaStream_t (NULL = legacy default stream).  Asynchronous.
 * CUDA graphs: a run may be captured into a graph and replayed when its K
 * split is 1 (MXA2A_INFO_SPLITS, or MXA2A_OPT_SPLIT_K = 1); with a split the
 * call returns MXA2A_ERR_CAPTURE_SPLIT while the stream is capturing, since
 * the partial tiles are tagged with the run's launch index, which a replay
 * does not change.  Replays share that index: a device time-out in one of
 * them stays reported (mxa2a_get_status) for the later ones, and
 * mxa2a_kernel_times does not see replays.
 * Errors: MXA2A_ERR_NULL_PTR, MXA2A_ERR_MISALIGNED, MXA2A_ERR_WRONG_DEVICE,
 * MXA2A_ERR_CAPTURE_SPLIT, MXA2A_ERR_CUDA (a launch failed); device
 * time-outs later through mxa2a_get_status.
 * Passage: all_to_all_matmul_impl.h, the kernel entry
 * AllToAllQuantMatmulKernelE4M3E4M3(shmemSpace, aGM, scaleAGM, bGM, scaleBGM,
 * cGM, tilingData), which runs Init and then Process: AllToAllProcess stages
 * the segments through the ring, MatmulProcess runs the block-scaled GEMM on
 * each staged slot.  The plan stands in for shmemSpace and tilingData.
 */
int mxa2a_run(mxa2a_plan *plan, const void *const *A_seg, const void *const *A_scale_seg, const void *B,
              const void *B_scale, void *C_bf16, void *stream);

/*
 * The direct-read variant (an ablation of the exchange): the GEMM reads each
 * A_seg[r] in place with TMA, as the all_to_all_matmul kernel reads its own
 * rank's block from local memory rather than from the receive buffer
 * (all_to_all_matmul_impl.h, MatmulProcess / LocalParams); there is no
 * staging ring, no credit protocol and no pack of A.  Its prologue packs the A
 * and B scales.  Same arguments and result bits as mxa2a_run_unfused with the
 * same K split; the single-CTA kernel only (MXA2A_ERR_INVALID_OPTION with
 * MXA2A_OPT_CTA_PAIR = 1).  The tensor maps of the segments are encoded on the
 * host and copied into the plan's workspace on the stream whenever the
 * segment pointers differ from the previous direct run.  The CUDA-graph rules
 * of mxa2a_run apply (MXA2A_INFO_SPLITS_UNFUSED).
 */
int mxa2a_run_direct(mxa2a_plan *plan, const void *const *A_seg, const void *const *A_scale_seg, const void *B,
                     const void *B_scale, void *C_bf16, void *stream);

/*
 * The unfused comparison path: first pack the R segments into one [M][K]
 * operand (and its scales), then run the same GEMM on it.  Same arguments;
 * the same result bits as mxa2a_run when both paths use the same K split
 * (MXA2A_OPT_SPLIT_K forces one; by default each path picks its own).
 * The CUDA-graph rules of mxa2a_run apply (MXA2A_INFO_SPLITS_UNFUSED).
 * Errors as for mxa2a_run.
 * Passage: all_to_all_matmul_impl.h, MatmulProcess (the QuantMatmulMxKernelSwat
 * GEMM over the received A) run only after AllToAllProcess has finished every
 * step (all_to_all_comm_udma.h, PutToAllRanks): the exchange and the GEMM in
 * sequence instead of overlapped, the comparison the method's own pipeline
 * is built to beat.
 */
int mxa2a_run_unfused(mxa2a_plan *plan, const void *const *A_seg, const void *const *A_scale_seg, const void *B,
                      const void *B_scale, void *C_bf16, void *stream);

/*
 * End-to-end variant with HOST buffers (same layouts): copies the inputs to
 * plan-owned device buffers (allocated on the first call), runs the fused
 * path and copies C back, all asynchronously on stream; the caller
 * synchronises the stream before reading C_bf16.  Pinned host buffers
 * (page-locked, as cudaHostAlloc or cudaHostRegister give) are used through
 * their device addresses: pinned A segments and scales are read in place by
 * the fused kernel's staging copies (the exchange then comes from host
 * memory), pinned B and B_scale are copied by the SMs in one launch, and a
 * pinned C is written by the GEMM's epilogue itself, tile by tile, while the
 * GEMM runs; pageable buffers go through one DMA copy each.  With a pinned C
 * a plan whose fused path is on CTA pairs by the automatic choice
 * (MXA2A_OPT_CTA_PAIR = 2) runs this call on single CTAs, the host link
 * being the bound; the plan keeps its choice.  The host buffers must stay
 * unchanged until the stream has passed the run.  Errors as for mxa2a_run.
 * Passage: all_to_all_matmul.cpp (the launcher), InitData and the
 * aclrtMemcpy calls that move the inputs to the device before the launch and
 * the output back after it.
 */
int mxa2a_run_host(mxa2a_plan *plan, const void *const *A_seg_host, const void *const *A_scale_seg_host,
                   const void *B_host, const void *B_scale_host, void *C_bf16_host, void *stream);

/*
 * Copy the device status block to *out (synchronous; call after the runs'
 * stream is synchronised) and mark it read.  out->code is MXA2A_OK unless a
 * launch since the previous call reported a device error.  Returns
 * MXA2A_ERR_NULL_PTR, MXA2A_ERR_WRONG_DEVICE, MXA2A_ERR_CUDA (the copy
 * failed) or MXA2A_OK.
 * Passage: the performance optimisation guide, section 2.1 (deadlocks after
 * moving from barrier_all to wait/notify): a wait that never ends is found by
 * a watchdog time-out followed by a dump of where the signals stopped (a slot
 * stuck at 1: the consumer never saw it; stuck at 0: the producer never
 * notified).  Here every device wait is bounded, and the first one that runs
 * out records its role, step, segment, slot and counter values.
 */
int mxa2a_get_status(mxa2a_plan *plan, mxa2a_status *out);

/* Option keys for mxa2a_set_option / mxa2a_get_option. */
enum mxa2a_option {
    MXA2A_OPT_TIMEOUT_NS = 1,      /* limit of every device wait, ns (default 2e9) */
    MXA2A_OPT_SPLIT_K = 2,         /* 0 = automatic, s >= 1: split K into s segment groups */
    MXA2A_OPT_ZIGZAG = 3,          /* 1 (default): alternate n-tile direction per m-tile */
    MXA2A_OPT_ROTATE = 4,          /* 1: start each tile's K loop at a rotated segment (default 0) */
    MXA2A_OPT_RECORD_EVENTS = 5,   /* n >= 1: time the main GEMM kernel of each run, keeping the last n
                                      (n <= 4096) for mxa2a_kernel_times; 0 = off (default) */
    MXA2A_OPT_EXCHANGE_ONLY = 6,   /* 1: fused runs only stage A into the ring (needs buffer_num >= steps) */
    MXA2A_OPT_FAULT_SKIP_STEP = 7, /* test knob: never publish staging step k (-1 = off); waits then time out */
    MXA2A_OPT_GRID = 8,            /* cap on persistent CTAs (0 = one per SM) */
    MXA2A_OPT_CHUNK_BYTES = 9,     /* target staging copy chunk in bytes; 0 (default): automatic,
                                      about two staging steps' tasks for all copy workers, 4..16 KiB */
    MXA2A_OPT_CTA_PAIR = 10,       /* the CTA-pair kernel (256-row tiles, one tcgen05 cta_group::2 MMA
                                      stream per pair), usable when M/128 is even and, on the fused
                                      path, buffer_num covers the steps of a 256-row tile.  2 (default):
                                      the fused path on pairs when its staging window
                                      (buffer_num * commMSize rows) holds at least two pair tiles per
                                      resident pair and no 128-column tile is asked for (MXA2A_OPT_TILE_N),
                                      the unfused path on single CTAs; 1: both paths on
                                      pairs wherever usable; 0: the single-CTA kernel
                                      (MXA2A_INFO_CTA_PAIR / _UNFUSED give the choice) */
    MXA2A_OPT_GROUP_M = 11,        /* largest raster group of the unfused path, in m rows
                                      (128-row tiles, or tile pairs), default 16 (the fused path's
                                      group: MXA2A_OPT_GROUP_FUSED) */
    MXA2A_OPT_TILE_N = 13,         /* GEMM tile width: 0 (default: 256) or 128 / 256.  128 doubles the
                                      tiles for the rows in flight and overlaps each tile's epilogue
                                      with the next tile (two TMEM accumulators) */
    MXA2A_OPT_ELEM_TYPES = 14,     /* element formats of A and B, the four kernel entries of the
                                      all_to_all_matmul kernel (all_to_all_matmul_impl.h):
                                      0 (default) E4M3 x E4M3, 1 E5M2 x E5M2, 2 E4M3 x E5M2,
                                      3 E5M2 x E4M3.  Scales stay E8M0, one per 32 along K */
    MXA2A_OPT_STEP_CREDITS = 15,   /* 1: whole-step staging protocol, as the all_to_all_matmul kernel's
                                      AllToAllProcess / MatmulProcess (a slot's next step is copied once
                                      every reader finished the whole previous step; a reader waits for
                                      the whole step); 0 (default): per-segment credits */
    MXA2A_OPT_COPY_SKEW_NS = 16,   /* test knob: the copy workers of every 4th CTA wait this many ns
                                      before each copy task (0 = off, at most 1e6) */
    MXA2A_OPT_GROUP_FUSED = 17,    /* fused raster group in m-tiles, n-tile outer inside a group
                                      (0, default: the m-tiles of buffer_num / 2 staging steps, at least
                                      one step; 1: m-tile by m-tile).  Rounded to a divisor of a
                                      staging step's m-tiles, or to a multiple of them within the
                                      ring's rows (buffer_num * commMSize); ignored when commMSize is
                                      not a multiple of 128 (with the CTA-pair kernel: 256, the group
                                      then counted in pairs of m-tiles) (the planner's choice:
                                      MXA2A_INFO_GROUP_FUSED, in m rows) */
    MXA2A_OPT_TAIL_SPLIT = 18,     /* 1 (default): when a path's tiles fill the persistent grid (its CTAs,
                                      or CTA pairs) more than once and the last round holds at most half
                                      the grid's worth, split that round's tiles in two along K (R even,
                                      K >= 8192; each half reads R / 2 segments, the sums done by the
                                      kernel as with MXA2A_OPT_SPLIT_K) so that twice as many CTAs share
                                      it; 0: whole tiles.  Only without a uniform split; a run under
                                      CUDA-graph capture leaves its tail whole (MXA2A_INFO_TAIL_SPLIT) */
    /* read-only plan facts (mxa2a_get_option only) */
    MXA2A_INFO_STEPS = 100,        /* M / commMSize */
    MXA2A_INFO_MTILES = 101,
    MXA2A_INFO_NTILES = 102,
    MXA2A_INFO_SPLITS = 103,       /* effective K split of the fused path */
    MXA2A_INFO_ITEMS = 104,        /* work items of the fused persistent GEMM */
    MXA2A_INFO_GRID_FUSED = 105,
    MXA2A_INFO_GRID_UNFUSED = 106,
    MXA2A_INFO_COPY_TASKS = 107,
    MXA2A_INFO_ROWS_PER_CHUNK = 108,
    MXA2A_INFO_WORKSPACE_BYTES = 109,
    MXA2A_INFO_SM_COUNT = 110,
    MXA2A_INFO_LAUNCHES = 111,     /* kernels launched by the last run call */
    MXA2A_INFO_SPLITS_UNFUSED = 112, /* effective K split of the unfused path */
    MXA2A_INFO_CTA_PAIR = 113,     /* 1 if the fused path runs the CTA-pair kernel */
    MXA2A_INFO_CTA_PAIR_UNFUSED = 114, /* 1 if the unfused path runs the CTA-pair kernel */
    MXA2A_INFO_GROUP_FUSED = 115,  /* raster group of the fused path (m rows) */
    MXA2A_INFO_GROUP_UNFUSED = 116, /* raster group of the unfused path (m rows) */
    MXA2A_INFO_TILE_N_FUSED = 117,  /* tile width of the fused path (128 or 256) */
    MXA2A_INFO_TILE_N_UNFUSED = 118, /* tile width of the unfused path (128 or 256) */
    MXA2A_INFO_KIND = 119,         /* enum mxa2a_kind */
    MXA2A_INFO_TAIL_SPLIT = 120,   /* K split of the fused path's last-round tiles (1: none) */
    MXA2A_INFO_TAIL_SPLIT_UNFUSED = 121 /* the same for the unfused path */
};

/* Set a tunable (MXA2A_OPT_*) or read it back, or read a plan fact
 * (MXA2A_INFO_*, read-only).  Returns MXA2A_ERR_INVALID_OPTION for an unknown
 * key, a value out of range, or a set of an MXA2A_INFO_* key; changing the
 * tiling re-derives the plan (and may reallocate its split-K scratch:
 * MXA2A_ERR_CUDA if that fails).
 * Passage: all_to_all_matmul.cpp (the launcher), the knobs it marks for
 * change, [MODIFY C1] bufferSize and [MODIFY C2] headMSize, and the
 * performance optimisation guide, sections 1.2 to 1.4 (core flattening and
 * split, signal granularity, swizzled tile order), whose choices the options
 * expose. */
int mxa2a_set_option(mxa2a_plan *plan, int key, int64_t value);
int mxa2a_get_option(mxa2a_plan *plan, int key, int64_t *value);

/* The planner alone, on the host (no device, nothing allocated): the choices
 * an all-to-all plan of this shape would make on a device with sm_count SMs
 * on which max_pairs_fused / max_pairs_unfused CTA pairs of the fused /
 * unfused pair kernel fit at once (a GB300: 152, 76, 76), with the planner
 * options opt_keys[i] = opt_values[i] (i < n_opts; MXA2A_OPT_SPLIT_K, _GRID,
 * _CHUNK_BYTES, _CTA_PAIR, _GROUP_M, _TILE_N, _ELEM_TYPES, _STEP_CREDITS,
 * _COPY_SKEW_NS, _GROUP_FUSED, _TAIL_SPLIT) applied in order.  Writes
 * info_values[i] = the value mxa2a_get_option would give for info_keys[i]
 * (i < n_info; any MXA2A_INFO_* or MXA2A_OPT_* key but MXA2A_INFO_WORKSPACE_BYTES
 * and MXA2A_INFO_LAUNCHES).  Returns the shape's mxa2a_validate code,
 * MXA2A_ERR_NULL_PTR for a missing array, MXA2A_ERR_INVALID_OPTION for a bad
 * device description, option or key (the outputs then partly written).
 * Passage: the performance optimisation guide, section 1.2 (fill all cores:
 * flattening and splitting the tiles over the cores), whose rules the planner
 * applies; it is how those rules are checked without a device. */
int mxa2a_plan_preview(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num,
                       int sm_count, int max_pairs_fused, int max_pairs_unfused, const int *opt_keys,
                       const int64_t *opt_values, int n_opts, const int *info_keys, int64_t *info_values,
                       int n_info);

/* Duration of the main GEMM kernel of the last run, in ms (needs
 * MXA2A_OPT_RECORD_EVENTS >= 1; synchronises on that run's end event).
 * Passage: all_to_all_matmul.cpp (the launcher), perf mode: the main kernel
 * timed alone, each round synchronised, after an L2 flush. */
int mxa2a_last_kernel_ms(mxa2a_plan *plan, float *ms);

/* Durations (ms) of the main GEMM kernel of the last min(max_count, recorded)
 * runs, oldest first, timed with CUDA events on each run's stream; *count
 * receives how many were written.  Synchronises on those runs' end events. */
int mxa2a_kernel_times(mxa2a_plan *plan, float *ms, int max_count, int *count);

/* Workspace regions readable with mxa2a_read_workspace (debug and tests). */
enum mxa2a_workspace {
    MXA2A_WS_RING = 1,      /* staging ring  [buffer_num][R][commMSize][kPerRank] */
    MXA2A_WS_SFA = 2,       /* A scales in MMA atom layout [K/128][ceil(M/128)][512] */
    MXA2A_WS_SFB = 3,       /* B scales in MMA atom layout [K/128][2*ceil(N/256)][512] */
    MXA2A_WS_FLAGS = 4,     /* credit counters, u64, one per 128-byte line */
    MXA2A_WS_APACKED = 5    /* unfused packed A [M][K] */
};

/* Synchronous copy of a workspace region to host memory (at most bytes);
 * *bytes_out receives the region's full size.  Synchronise the plan's
 * stream first.
 * Passage: all_to_all_matmul.cpp (the launcher), precision mode: the
 * communication buffer's A and scales are copied back (shmem_A.bin,
 * shmem_scale.bin) to check the exchange by itself. */
int mxa2a_read_workspace(mxa2a_plan *plan, int which, void *host_dst, size_t bytes, size_t *bytes_out);

/* Benchmark helper: add 1 to every 32-bit word of a device buffer (bytes %
 * 16 == 0), evicting other data from L2 when bytes exceeds its size.
 * Passage: all_to_all_matmul.cpp (the launcher), perf mode: heavy_add_kernel
 * over a cache-flush buffer larger than L2 before every timed round. */
int mxa2a_l2_flush(void *device_buf, size_t bytes, void *stream);

/*
 * The fused path for callers that cannot allocate device memory — a runtime
 * whose device memory is entirely budgeted by its own pool allocator (a
 * library's cudaMalloc can fail or fragment it there), or a latency-critical
 * loop where cudaMalloc / cudaFree would implicitly synchronise the device.
 * The pages have no counterpart of this entry point; it is a deployment
 * variant of mxa2a_run.
 *
 * Same shape rules, data layouts and result as mxa2a_run with E4M3 x E4M3
 * operands (the element-type option of a plan does not exist here), run on
 * the single-CTA kernel with no K split: the result bits equal those of
 * mxa2a_run of a plan with MXA2A_OPT_SPLIT_K = 1, MXA2A_OPT_CTA_PAIR = 0
 * and MXA2A_OPT_TAIL_SPLIT = 0.
 * It allocates nothing: the staging ring, scale tiles, credit
 * counters and status block live in one static device array of 16 MiB that
 * every GPU which loads this library holds until the process exits.  A shape
 * whose ring + scale tiles + counters exceed it returns
 * MXA2A_ERR_SCRATCH_TOO_SMALL before any device work (the ring alone is
 * buffer_num * R * commMSize * kPerRank bytes).  The first call on a device
 * looks up the array's device address once; make that first call before any
 * stream capture begins.  Every call reuses the same array (the counters are
 * cleared on the stream at the start of each call), so calls that overlap on
 * the GPU — on two streams, or from two host threads — race.  Device-side
 * wait time-outs are not reported by this entry point: the kernel then stops
 * early, C is left partly written (undefined), and the call has already
 * returned MXA2A_OK.  Only a lost staging credit can cause one, i.e. a
 * defect, not an input.  Asynchronous on
 * stream (a cudaStream_t, NULL = legacy default stream).
 */
int mxa2a_run_noalloc(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num,
                      const void *const *A_seg, const void *const *A_scale_seg, const void *B, const void *B_scale,
                      void *C_bf16, void *stream);

/* Free the plan's workspace (synchronises the device first). NULL is a no-op.
 * Passage: all_to_all_matmul.cpp (the launcher), the teardown after the
 * runs (aclshmem_free of the communication space, aclrtFree of the buffers). */
void mxa2a_destroy(mxa2a_plan *plan);

/* Static string for an error code (never NULL; unknown codes get a generic
 * text).  Passage: all_to_all_matmul.cpp (the launcher), the messages its
 * argument checks throw ("ERROR: k must be divisible by rankNum", ...). */
const char *mxa2a_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MXA2A_H */

// Shared declarations between the CUDA kernels and the C-ABI host layer of
// libmxa2a (fused AllToAll + MXFP8 block-scaled GEMM on sm_103a).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxa2a {

constexpr int kMaxSegments = 64;   // R limit (segment pointer tables live in kernel params)

// GEMM tile per CTA: 128 rows (M) x BN columns (N), 128-byte (= 128 FP8) K
// blocks, with BN = 256 (the wide tile) or 128 (the narrow tile: twice the
// tiles for a given rows-in-flight, and two TMEM accumulators so a tile's
// epilogue overlaps the next tile's MMAs).  In the CTA-pair variant two CTAs
// compute a 256 x 256 tile with one tcgen05 cta_group::2 MMA stream, each
// holding half of B, so a stage is smaller and the ring deeper.
constexpr int BM = 128;
constexpr int BN = 256;            // the wide tile (also the padding unit of the B scale atoms)
constexpr int BN_NARROW = 128;
constexpr int BK = 128;
constexpr int kStagesSingle = 4;   // wide tile: 49.5 KiB stages
constexpr int kStagesNarrow = 6;   // narrow tile: 33 KiB stages
constexpr int kStagesPair = 6;
constexpr int kMaxStages = 6;
constexpr int kMaxAccBufs = 2;
constexpr int kThreads = 512;      // 16 warps (4 per SM sub-partition: 128 registers each), roles below
constexpr int kWarpTma = 0;        // TMA producer 0 (one elected lane): even stages
constexpr int kWarpMma = 1;        // TMEM allocator + MMA issuer (one elected lane)
constexpr int kWarpEpi0 = 2;       // warps 2..9: epilogue, warp w drains TMEM lane quarter w%4,
constexpr int kEpiWarps = 8;       //   column half (w-2)/4 of the accumulator
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kWarpCopy0 = 10;     // warps 10, 11, 14, 15: staging copy workers, one per warp
constexpr int kCopyWarps = 4;      //   (fused kernel only; idle in the unfused kernel)
constexpr int kWarpTma1 = 12;      // TMA producer 1 (one elected lane): odd stages
// Warp 13 is no copy worker: it would share an SM sub-partition (warp % 4)
// with the MMA-issuing warp 1, and a busy copy warp there slows the MMA issue.
// In the fused kernel one of its lanes returns the staging credits (mostly
// asleep), so that the MMA thread issues no global atomics.
__host__ __device__ constexpr bool is_copy_warp(int w) { return w == 10 || w == 11 || w >= 14; }
constexpr int kWarpCredit = 13;
// One thread's TMA loads overlap poorly (about one stage per 0.4 us per
// thread on this GPU); two issuing warps double the per-SM load rate.
constexpr int kProducers = 2;

constexpr int kAStageBytes = BM * BK;        // 16 KiB
constexpr int kSfAtomBytes = 512;            // 128 rows x 4 E8M0 bytes (one 128-K block)
constexpr int kSfaStageBytes = kSfAtomBytes;
constexpr int kEpiBufBytes = 32 * 32 * 2;    // per epilogue warp: one 32x32 BF16 chunk of C

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemAccCol = 0;          // accumulators: 1 x 256 (wide) or 2 x 128 (narrow) fp32 columns
constexpr uint32_t kTmemSfCol = 256;         // per stage: 4 SFA + 4 per 128 B columns
constexpr int kWarpSf0 = 6;                  // single-CTA kernel: epilogue warps 6..9 (lane quarters 2, 3,
constexpr int kSfWarps = 4;                  //   0, 1) also write each stage's scale factors into TMEM

// Device error codes written to the status block (same numbers as the C ABI).
constexpr int kErrTimeout = 6;
constexpr int kErrDeviceCheck = 8;

// Role ids recorded with a device error.
constexpr int kRoleCopy = 1, kRoleTma = 2, kRoleMma = 3, kRoleEpi = 4, kRoleExit = 5, kRoleReduce = 6;

struct DevStatus {
    unsigned long long key;   // (launch_id << 8) | code, first error of a launch wins
    int role, block, step, segment, slot, pad;
    long long observed, expected;
};

// Monotonic credit counters of the staging ring, each on its own 128-byte line.
// filled[slot][r]:  staging copy chunks published for (slot, segment r)
// drained[slot][r]: work items that finished reading segment r of the slot
// staged[slot]:     chunks of all segments of the slot published; lets a
//                   reader check a whole step with one load
// cta_done:         CTAs that reached the end (the last one zeroes everything)
// copy_next:        next staging copy task to claim (tasks are claimed in order)
// sfb_done:         CTAs that finished their slice of the B scale pack (kernel prologue)
struct FlagLayout {
    static constexpr int kLine = 16;  // 16 x u64 = 128 bytes
    __host__ __device__ static size_t filled(int slot, int r, int R) { return (size_t)(slot * R + r) * kLine; }
    __host__ __device__ static size_t drained(int slot, int r, int bn, int R) {
        return (size_t)(bn * R + slot * R + r) * kLine;
    }
    __host__ __device__ static size_t staged(int slot, int bn, int R) { return (size_t)(2 * bn * R + slot) * kLine; }
    __host__ __device__ static size_t cta_done(int bn, int R) { return (size_t)(2 * bn * R + bn) * kLine; }
    __host__ __device__ static size_t copy_next(int bn, int R) { return (size_t)(2 * bn * R + bn + 1) * kLine; }
    __host__ __device__ static size_t sfb_done(int bn, int R) { return (size_t)(2 * bn * R + bn + 2) * kLine; }
    __host__ __device__ static size_t words(int bn, int R) { return (size_t)(2 * bn * R + bn + 3) * kLine; }
};

struct GemmParams {
    int R, M, N, ka, K, cm, bn, steps;
    int Mt, Nt, S, W;           // m-tiles, n-tiles, K splits, work items
    // tail split (S == 1, single-CTA kernel): items W_dp .. W-1 are the last
    // (W - W_dp) / S_tail tiles, each split S_tail ways in K; W_dp = W: none
    int W_dp, S_tail;
    int pair;                   // 1: CTA-pair kernel, work items are pairs of m-tiles (Mt even)
    int tile_n;                 // BN of this launch: 256 or 128 (Nt = ceil(N / tile_n))
    int fmt_a, fmt_b;           // element formats (MMA type codes): 0 E4M3, 1 E5M2
    int kb_per_seg;             // ka / 128
    int Mg, Ng2;                // 128-row groups of A (scale atoms), 128-col groups of B (padded to 256)
    int box_m;                  // rows per A TMA box: 128 or 64
    int zigzag, rotate;
    int group_m;                // m rows (tiles, or tile pairs) per raster group
    const uint8_t* sfa;         // A scales, MMA atom layout [K/128][Mg][512]
    const uint8_t* sfb;         // B scales, MMA atom layout [K/128][Ng2][512]
    // sfb_inline: the kernel's prologue packs B_scale ([N][K/32] E8M0) into sfb
    // (every CTA a slice, counted on the sfb_done flag) instead of a separate
    // pack kernel; needs all CTAs resident (cooperative launch)
    int sfb_inline;
    const uint8_t* B_scale;
    // direct (unfused kernel only): A is read in place from the R segment
    // buffers through seg_maps[r] (tensor maps in global memory, 64-byte
    // aligned), and the prologue also packs the A scales into sfa
    int direct;
    const CUtensorMap* seg_maps;
    uint16_t* C;                // bf16 [M][N]
    uint16_t* c_host;           // non-null: C goes to this host buffer (its device view) instead, by
                                // generic stores from the epilogue (no reduce-scatter routing then)
    // split-K (S > 1, or a tail item): every split writes its fp32 tile to
    // partial[slot][q] ([BM][BN]) and publishes ready[slot][q] = launch_id;
    // once all splits have, split q sums its share of the tile's units, the
    // splits in order, and writes C.  slot: the tile (mt * Nt + nt) under a
    // uniform split, its place among the tail's tiles for a tail item.
    float* partial;             // fp32 [slots][S][tile_n/4][BM][4] (4-column chunks, row-contiguous)
    unsigned long long* ready;  // [slots][S]
    // fused staging
    int fused, exchange_only;
    int rows_per_chunk, chunks_per_seg, n_copy_tasks;
    int fault_skip_step;        // test knob: never publish the fill of this step (-1 = off)
    int step_credits;           // 1: whole-step fill and release (the pages' per-step protocol)
    int copy_skew_ns;           // test knob: copy workers of every 4th CTA wait this long before each task
    uint8_t* ring;              // [bn][R][cm][ka]
    uint8_t* sfa_stage;         // writable alias of sfa (staged by the copy role)
    unsigned long long* flags;
    DevStatus* status;
    unsigned long long launch_id;
    long long timeout_ns;
    // seg_rows: 0 for the all-to-all (A_seg[r] holds K slice r of all M rows,
    // [M][ka]); > 0 for the all-gather (A_seg[j] holds rows j*seg_rows ..
    // (j+1)*seg_rows-1 of A with all K = R*ka columns, [seg_rows][K]; the R
    // K slices are then column ranges of every block)
    int seg_rows;
    const uint8_t* A_seg[kMaxSegments];
    const uint8_t* A_sf_seg[kMaxSegments];
    // GEMM + ReduceScatter (rs_rows > 0, S == 1, the kernel without staging):
    // the output rows form rs_R blocks of rs_rows.  The epilogue stores block
    // j != rs_rank, rounded to BF16, through send_maps[j] (bf16 [rs_rows][N],
    // 64-byte aligned maps in global memory) and block rs_rank through tmap_c
    // (C = out, [rs_rows][N]), then counts its warp in rs_cnt[tile]; the copy
    // warps then sum each row of out with recv[j] (fp32, j in order) in place.
    // The m-tiles are taken starting at block rs_rank's, so its sums overlap
    // the other blocks' GEMM.
    // GEMM + AllReduce (one-shot) uses the same path with one block of all M
    // rows (rs_own = 0) and rs_publish = 1: the block's partial goes to
    // send_maps[0] (the buffer the peers read, rs_pub) and the sums read it
    // there and write out.  rs_rank is the rank's place in the sum; rs_own the
    // block summed here (RS: rs_rank).
    int rs_rows, rs_rank, rs_R, rs_own, rs_publish;
    const CUtensorMap* send_maps;
    const uint16_t* recv[kMaxSegments];
    const uint16_t* rs_pub;
    unsigned long long* rs_cnt;   // [Mt * Nt], zero between launches
};

// Where row m of K slice r of the stacked A lives: its input buffer and the
// row inside it; seg_ld is that buffer's row length in bytes (scales: /32)
// and seg_col0 the column where slice r starts in it.
struct SegRow {
    int seg, row;
};
__host__ __device__ inline SegRow seg_row(const GemmParams& p, int r, int m) {
    if (p.seg_rows > 0) {
        const int j = m / p.seg_rows;
        return {j, m - j * p.seg_rows};
    }
    return {r, m};
}
__host__ __device__ inline int seg_ld(const GemmParams& p) { return p.seg_rows > 0 ? p.K : p.ka; }
__host__ __device__ inline int seg_col0(const GemmParams& p, int r) { return p.seg_rows > 0 ? r * p.ka : 0; }

// Launchers (mxgemm.cu / aux_kernels.cu).  All return cudaError_t of the launch.
// tmap_c: C as bf16 [M][N], box 32 rows x 32 columns, 64-byte swizzle (the epilogue's TMA stores)
// tmap_sf: the A and B scale atoms ([K/128][Mg][512] and [K/128][Ng2][512] u8)
// as 2D u8 tensors of 256-byte rows, boxes of 2 and 4 rows (one atom, two
// atoms); needed by the CTA-pair kernel, whose odd CTA's loads complete on the
// even CTA's barrier (a form the plain bulk copy lacks), else may be NULL
cudaError_t launch_mxgemm(const GemmParams& p, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                          const CUtensorMap& tmap_c, int grid, bool fused, cudaStream_t stream,
                          const CUtensorMap* tmap_sf = nullptr);
// CTA pairs of the pair kernel that can be resident at once (0 if it cannot run)
int mxgemm_max_pairs(bool fused);
cudaError_t launch_pack_a(const GemmParams& p, uint8_t* a_packed, int grid, cudaStream_t stream);
cudaError_t launch_pack_sfb(const uint8_t* B_scale, int N, int K, int Ng2, uint8_t* sfb, cudaStream_t stream);
cudaError_t launch_l2_flush(void* buf, size_t bytes, cudaStream_t stream);
// The reduce-scatter of the unfused GEMM + ReduceScatter: P bf16 [R*rows][N];
// send[j] = block j of P (j != rank); out = bf16(sum over j in order of block
// rank of P (j == rank) or recv[j]), fp32 adds.  Pointer arrays of R entries.
// With nblk blocks of rows (RS: nblk = R, own = rank; one-shot all-reduce:
// nblk = 1, own = 0, P is the published partial).
struct RsArgs {
    const uint16_t* P;
    const uint16_t* recv[kMaxSegments];
    uint16_t* send[kMaxSegments];
    uint16_t* out;
    int R, rank, rows, N, nblk, own;
};
cudaError_t launch_rs_reduce(const RsArgs& a, cudaStream_t stream);

}  // namespace mxa2a

// Persistent warp-specialised MXFP8 block-scaled GEMM for sm_103a, with an
// optional fused staging ("AllToAll") role.
//
// The operation is the one of the all_to_all_matmul kernel
// (all_to_all_matmul_impl.h, AllToAllProcess + MatmulProcess): the R
// K-segments of A are staged block by block (commMSize rows per step) into a
// ring of buffer_num slots (all_to_all_comm_udma.h, PutSegmentToRank: segment
// r of a step lands at r*commMSize*kPerRank inside the slot), a producer
// publishes each filled slot, the GEMM consumes it with split-K over the
// segments and returns the slot's credit.  On one GPU the segments are R
// separate HBM buffers and the "exchange" is this kernel's own copy role.
//
// CTA roles (512 threads = 16 warps, one CTA per SM, persistent over work items):
//   warps 0, 12  TMA producers (even / odd stages): wait for a slot's segment
//            to be published, then stream A (from the ring, or from the packed
//            A when unfused), B and both scale tiles into a shared-memory ring
//            of stages (the scale tiles on their own barrier in the single-CTA
//            kernel).  Two issuing warps: one thread's TMA loads overlap
//            poorly, two reach about twice the per-SM load rate.
//   warp 1   TMEM owner and MMA issuer: 4 tcgen05.mma kind::mxf8f6f4
//            block-scaled MMAs (128x256x32 each) per 128-wide K block.
//            In the CTA-pair kernel the even CTA issues 256x256x32 MMAs for
//            both CTAs (.cta_group::2), copying each stage's scale factors to
//            TMEM first (tcgen05.cp); the odd CTA's loads complete on the even
//            CTA's barriers and its epilogue warps release the accumulator
//            there, so the odd CTA's warp 1 only owns its TMEM.
//   warps 2-9 epilogue: TMEM -> registers -> BF16 -> shared staging -> TMA
//            store, or, for split K, the in-kernel fixed-order reduction of
//            the split partials.  Warp w drains TMEM lane quarter w%4, column
//            half (w-2)/4.  In the single-CTA kernel warps 6-9 (one per lane
//            quarter) also write each stage's scale factors into TMEM
//            (tcgen05.st) as soon as they land, ahead of the stage's A and B.
//   warps 10, 11, 14, 15 staging copy (fused only): four independent workers
//            per CTA take copy tasks (step, segment, chunk) in step order,
//            wait for the slot's credit, copy the rows of A_seg[r] and their
//            scales, publish.  (Warp 13 idles: it would share an SM
//            sub-partition with the MMA issuer.)  In the kernel without
//            staging these warps sum a GEMM + ReduceScatter's (or one-shot
//            AllReduce's) own rows with the received partials once the
//            epilogue has stored them.
//
// Prologue: every CTA packs a slice of the B scales into MMA atoms (and, for
// the direct read, of the A scales) and counts itself on a grid counter that
// the producers wait for (the launch is cooperative); in the fused kernel the
// copy warps skip the pack and start staging at once.
//
// The same kernels serve the sibling operators: the all-gather stages row
// blocks in K slices (the input buffer and column of a slice come from
// seg_row / seg_ld / seg_col0), and the reduce-scatter and all-reduce route
// each finished tile in the epilogue (peers' rows to their send buffers, the
// own rows or the published partial through a tensor map each).
//
// Credits (the pages' per-slot signals with credit return, performance guide
// 1.1/1.3, kept per segment as its fine-grained signals suggest) are
// monotonic u64 counters: segment r of a slot holds step s once
// filled[slot][r] >= (s/bn + 1) * chunks_per_seg, and may be overwritten by
// step s once drained[slot][r] counts every reader of segment r of the
// earlier steps that used the slot.  A reader returns a segment's credit as
// soon as its TMA loads of that segment have landed, so the next step's copy
// of segment r overlaps the readers' work on the later segments.  Nothing is
// reset inside a launch; the last CTA to finish zeroes the counters for the
// next launch.  Every wait is bounded by a time limit and reports through the
// status block instead of hanging.
#include <cuda_bf16.h>

#include <cstring>

#include "atoms.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa2a {
using namespace ptx;

// Optional event trace (built only with -DMXA2A_TRACE): per CTA, up to
// kTraceCap (event, %globaltimer) pairs; event = kind << 56 | a << 28 | b.
#ifdef MXA2A_TRACE
constexpr int kTraceCtas = 160;
constexpr int kTraceCap = 4096;
__device__ unsigned long long g_trace[kTraceCtas * kTraceCap * 2];
__device__ unsigned g_trace_n[kTraceCtas];
__shared__ unsigned s_trace_n;
__device__ __forceinline__ void trace_ev(unsigned kind, unsigned a, unsigned b) {
    if (blockIdx.x >= kTraceCtas) return;
    const unsigned i = atomicAdd(&s_trace_n, 1u);
    if (i >= kTraceCap) return;
    unsigned long long* e = g_trace + ((size_t)blockIdx.x * kTraceCap + i) * 2;
    e[0] = ((unsigned long long)kind << 56) | ((unsigned long long)(a & 0xFFFFFFFu) << 28) | (b & 0xFFFFFFFu);
    e[1] = globaltimer();
}
#define TRACE(k, a, b) trace_ev((k), (unsigned)(a), (unsigned)(b))
#else
#define TRACE(k, a, b) ((void)0)
#endif

// In the CTA-pair kernel the even CTA's full[] barriers cover both CTAs'
// loads of a stage (its producer arms them for the bytes of both CTAs; every
// TMA load of either CTA completes on them), and its acc_empty[] barriers
// count the epilogue warps of both CTAs; the odd CTA's copies of those
// barriers are unused.  tx_own[s]: the bytes this CTA's producer loaded into
// stage s last; tx_odd[s] (even CTA): the odd CTA's bytes it armed stage s for.
// (acc_empty: count 2 * kEpiWarps, one arrival per epilogue warp of each CTA.)
struct __align__(8) SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[kMaxAccBufs];    // per TMEM accumulator buffer
    uint64_t acc_empty[kMaxAccBufs];
    uint64_t sf_loaded[kMaxStages];    // single-CTA kernel: the stage's scale atoms have landed in smem
    uint64_t sf_ready[kMaxStages];     // single-CTA kernel: the scale warps wrote them into TMEM
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort;
    volatile int issued[kProducers];   // per producer: 1 + index of its last issued stage
    volatile uint32_t tx_own[kMaxStages];
    volatile uint32_t tx_odd[kMaxStages];
    volatile int consumed;   // stages whose full barrier the MMA thread has passed
};

// Per kernel variant (CTA pair or not, tile width kBN): pipeline depth, stage
// sizes, TMEM use, and the shared-memory layout of one CTA:
// [A stages][B stages][SFA stages][SFB stages][C staging][control]
template <bool kPair, int kBN>
struct Lay {
    static_assert(kBN == BN || (kBN == BN_NARROW && !kPair), "tile width");
    static constexpr int kStg = kPair ? kStagesPair : (kBN == BN ? kStagesSingle : kStagesNarrow);
    static constexpr int kBRows = kPair ? kBN / 2 : kBN;     // rows of B this CTA loads per stage
    static constexpr int kBStage = kBRows * BK;
    static constexpr int kSfbAtoms = kBN / 128;              // B scale atoms of the tile's columns (each
                                                             // CTA of a pair needs all of them in its TMEM)
    static constexpr int kSfbStage = kSfbAtoms * kSfAtomBytes;
    static constexpr int kAccBufs = kBN == BN_NARROW ? 2 : 1;   // TMEM accumulators (512 columns hold
                                                                 // 2 x 128 + scales, not 2 x 256 + scales)
    static constexpr uint32_t kSfCols = 4 + 4 * kSfbAtoms;   // TMEM scale columns per stage
    static constexpr size_t A = 0;
    static constexpr size_t B = A + (size_t)kStg * kAStageBytes;
    static constexpr size_t Sfa = B + (size_t)kStg * kBStage;
    static constexpr size_t Sfb = Sfa + (size_t)kStg * kSfaStageBytes;
    static constexpr size_t Epi = Sfb + (size_t)kStg * kSfbStage;   // one C staging buffer per epilogue warp
    static constexpr size_t Ctl = Epi + (size_t)kEpiWarps * kEpiBufBytes;
    static constexpr size_t Total = Ctl + sizeof(SmemCtl) + 1024;   // + runtime 1 KiB alignment
    static_assert(Total <= 227 * 1024, "shared memory");
    static_assert(kStg <= kMaxStages && kAccBufs <= kMaxAccBufs, "barrier arrays");
    static_assert(kAccBufs * kBN <= (int)kTmemSfCol && kTmemSfCol + kStg * kSfCols <= kTmemCols, "TMEM columns");
    static_assert(Epi % 1024 == 0, "C staging buffers need 512-byte alignment for the 64-byte swizzle");
    static_assert((size_t)kStg * kAStageBytes >= (size_t)kTileWords * 4, "the prologue's pack tile fits the A stages");
};

// ------------------------------------------------------------------ work items
struct Item {
    int mt, nt, q, seg_lo, nseg, rot;
    int S;      // K splits of this item's tile
    int tail;   // the tile's place among the split tail's tiles, or -1
};

// Flattened work id -> (m row, n-tile, K split), where the m row is an m-tile
// (or, in the CTA-pair kernel, a pair of m-tiles).  Items are rastered in
// groups of group_m m rows: group after group (so the staging steps are
// consumed in order), inside a group n-tile outer and m row inner (so the
// CTAs running at the same time share a few B tiles and a few A rows in
// L2), with the n direction reversed on odd groups (zigzag) so a group starts
// on the B tiles the previous one ended on.  On the fused path a group is
// whole staging steps that fit in the ring together.  The K split (S ways)
// is the innermost index; each item may start its K loop at a rotated
// segment.
__device__ __forceinline__ Item decode_tile(const GemmParams& p, int w, int S) {
    Item it;
    const int rows = p.pair ? p.Mt / 2 : p.Mt;
    const int per_group = p.group_m * p.Nt * S;
    const int g = w / per_group;
    const int gm = min(p.group_m, rows - g * p.group_m);     // m rows in this group
    const int rem = w - g * per_group;
    const int ntl = rem / (gm * S);
    const int rem2 = rem - ntl * (gm * S);
    it.mt = g * p.group_m + rem2 / S;
    // GEMM + ReduceScatter: start at the m-tile of this rank's first row
    if (p.rs_rows > 0 && !p.pair) it.mt = (it.mt + (p.rs_own * p.rs_rows) / BM) % p.Mt;
    it.q = rem2 % S;
    it.nt = (p.zigzag && (g & 1)) ? (p.Nt - 1 - ntl) : ntl;
    it.seg_lo = it.q * p.R / S;
    const int seg_hi = (it.q + 1) * p.R / S;
    it.nseg = seg_hi - it.seg_lo;
    it.rot = p.rotate ? (it.mt + it.nt) % it.nseg : 0;
    it.S = S;
    it.tail = -1;
    return it;
}

// Work id -> item.  Items before W_dp are whole tiles (or the uniform split's
// parts).  With a tail split, the tiles from W_dp on in the same order -- the
// ones the persistent grid's last, partly filled round would hold -- come as
// S_tail consecutive items each, split q reading segments q*R/S_tail ..
// (q+1)*R/S_tail - 1, so that the round's work spreads over more CTAs.
__device__ __forceinline__ Item decode_item(const GemmParams& p, int w) {
    if (w < p.W_dp || p.S_tail <= 1) return decode_tile(p, w, p.S);
    const int t = (w - p.W_dp) / p.S_tail;
    Item it = decode_tile(p, p.W_dp + t, 1);
    it.S = p.S_tail;
    it.tail = t;
    it.q = (w - p.W_dp) - t * p.S_tail;
    it.seg_lo = it.q * p.R / it.S;
    it.nseg = (it.q + 1) * p.R / it.S - it.seg_lo;
    it.rot = p.rotate ? (it.mt + it.nt) % it.nseg : 0;
    return it;
}

// The slot of a CTA's tile among the split partials: the tile itself under a
// uniform split, its place in the tail for a tail item (in a CTA pair, two
// slots per tail tile, one per CTA's m-tile).
__device__ __forceinline__ size_t split_slot(const GemmParams& p, const Item& item, int mt) {
    if (item.tail < 0) return (size_t)mt * p.Nt + item.nt;
    return p.pair ? 2 * (size_t)item.tail + (size_t)(mt - 2 * item.mt) : (size_t)item.tail;
}

// The m-tile a CTA works on for an item.
template <bool kPair>
__device__ __forceinline__ int cta_mtile(const Item& item, uint32_t rank) {
    return kPair ? 2 * item.mt + (int)rank : item.mt;
}

// First work item of this CTA (or CTA pair) and the stride between its items.
template <bool kPair>
__device__ __forceinline__ int first_item() {
    return kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
}
template <bool kPair>
__device__ __forceinline__ int item_stride() {
    return kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
}

// With the rows in one m-tile (M <= 128) every B scale atom is read by exactly
// one item (an item is an n-tile and a K range; a tile's K splits cover
// disjoint ranges), so each CTA of the single-CTA kernel packs the atoms its
// own items read, and its producers need no grid-wide count, only this CTA's
// barrier.
__device__ __forceinline__ bool own_sfb_pack(const GemmParams& p) {
    return p.sfb_inline && !p.direct && p.Mt == 1;
}

__device__ __forceinline__ int num_boxes(const GemmParams& p, int mt) {
    const int rows = min(BM, p.M - mt * BM);
    return (rows + p.box_m - 1) / p.box_m;
}

// Work items that read one segment of staging step s: the m-tiles overlapping
// its rows x Nt (of a tile's S split items exactly one covers the segment).
__device__ __forceinline__ unsigned long long readers_of_segment(const GemmParams& p, int s) {
    const int first = (s * p.cm) / BM;
    const int last = ((s + 1) * p.cm - 1) / BM;
    return (unsigned long long)(last - first + 1) * (unsigned long long)p.Nt;
}

// ------------------------------------------------------------------ errors and bounded waits
__device__ void record_error(const GemmParams& p, int code, int role, int step, int seg, int slot,
                             long long observed, long long expected) {
    DevStatus* st = p.status;
    const unsigned long long mine = (p.launch_id << 8) | (unsigned long long)code;
    unsigned long long cur = atomicAdd(&st->key, 0ull);
    for (;;) {
        if ((cur >> 8) == p.launch_id) return;   // this launch already reported
        const unsigned long long prev = atomicCAS(&st->key, cur, mine);
        if (prev == cur) break;
        cur = prev;
    }
    st->role = role;
    st->block = blockIdx.x;
    st->step = step;
    st->segment = seg;
    st->slot = slot;
    st->observed = observed;
    st->expected = expected;
    __threadfence();
}

__device__ __forceinline__ bool launch_failed(const GemmParams& p) {
    return (ld_relaxed_u64(&p.status->key) >> 8) == p.launch_id;
}

// Wait for an mbarrier phase; false on time-out or when the CTA is aborting.
// cluster: the phase is completed by arrivals from the other CTA of a pair
// (acquire at cluster scope).
__device__ __forceinline__ bool try_wait_scoped(uint64_t* bar, uint32_t parity, bool cluster) {
    return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}
__device__ bool wait_mbar(const GemmParams& p, SmemCtl* ctl, uint64_t* bar, uint32_t parity, int role,
                          bool cluster = false) {
    if (try_wait_scoped(bar, parity, cluster)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (try_wait_scoped(bar, parity, cluster)) return true;
        if (ctl->abort) return false;
        if ((n & 63) == 0) {
            if (globaltimer() - t0 > (uint64_t)p.timeout_ns) {
                record_error(p, kErrTimeout, role, -1, -1, -1, -1, (long long)parity);
                ctl->abort = 1;
                return false;
            }
            if (launch_failed(p)) {
                ctl->abort = 1;
                return false;
            }
        }
    }
}

// Whole-warp variant: every lane waits (each acquires), the outcome is uniform.
__device__ __forceinline__ bool wait_mbar_warp(const GemmParams& p, SmemCtl* ctl, uint64_t* bar, uint32_t parity,
                                               int role, bool cluster = false) {
    const bool ok = wait_mbar(p, ctl, bar, parity, role, cluster);
    return __all_sync(0xffffffffu, ok);
}

// Cleanup wait: only the time limit ends it (used after an abort).
__device__ void wait_mbar_plain(const GemmParams& p, uint64_t* bar, uint32_t parity, bool cluster = false) {
    const uint64_t t0 = globaltimer();
    while (!try_wait_scoped(bar, parity, cluster)) {
        if (globaltimer() - t0 > (uint64_t)p.timeout_ns) {
            record_error(p, kErrTimeout, kRoleExit, -1, -1, -1, -1, (long long)parity);
            return;
        }
    }
}

// Wait until a global credit counter reaches target (acquire).
__device__ bool wait_counter(const GemmParams& p, SmemCtl* ctl, const unsigned long long* ctr,
                             unsigned long long target, int role, int step, int seg, int slot) {
    unsigned long long v = ld_acquire_u64(ctr);
    if (v >= target) return true;
    const uint64_t t0 = globaltimer();
    uint32_t nap = 64;   // exponential back-off keeps many pollers off the counter's L2 line
    for (uint32_t n = 1;; ++n) {
        __nanosleep(nap);
        if (nap < 256) nap <<= 1;
        v = ld_acquire_u64(ctr);
        if (v >= target) return true;
        if (ctl->abort) return false;
        if ((n & 15) == 0) {
            if (globaltimer() - t0 > (uint64_t)p.timeout_ns) {
                record_error(p, kErrTimeout, role, step, seg, slot, (long long)v, (long long)target);
                ctl->abort = 1;
                return false;
            }
            if (launch_failed(p)) {
                ctl->abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over its threads: true for all of
// them only if every thread passed true.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ roles
template <bool kPair, int kBN>
__device__ void producer_role(const GemmParams& p, const CUtensorMap* tma, const CUtensorMap* tmb,
                              const CUtensorMap* tm_sfa, const CUtensorMap* tm_sfb, uint8_t* sA, uint8_t* sB,
                              uint8_t* sSfa, uint8_t* sSfb, SmemCtl* ctl, bool fused, uint32_t rank, int pid) {
    using L = Lay<kPair, kBN>;
    // CTA pair: every stage's loads of both CTAs complete on the even CTA's
    // full barrier, which each producer arms for its own bytes
    const uint32_t full0 = kPair ? mapa_shared(smem_u32(&ctl->full[0]), 0) : 0u;
    // B tiles are re-read by every m-tile: keep them in L2; A (ring or packed) is read by one
    // row of tiles at a time
    const uint64_t pol_keep = l2_policy_evict_last();
    const uint64_t pol_stream = l2_policy_evict_first();
    int it = 0;   // global stage sequence number; this producer issues it % kProducers == pid
    if (p.sfb_inline || p.direct) {
        // (all CTAs' atoms: the grid-wide count; only this CTA's own: its barrier, passed already)
        if ((kPair || !own_sfb_pack(p)) &&
            !wait_counter(p, ctl, p.flags + FlagLayout::sfb_done(p.bn, p.R), gridDim.x, kRoleTma, -1, -1, -1))
            return;
        fence_proxy_async_global();   // the atoms were written through the generic proxy; TMA reads them
        if (pid == 0) TRACE(23, 0, 0);
    }
    for (int w = first_item<kPair>(); w < p.W; w += item_stride<kPair>()) {
        const Item item = decode_item(p, w);
        const int mt = cta_mtile<kPair>(item, rank);
        const int nbox = fused ? num_boxes(p, mt) : 1;
        const uint32_t a_bytes = fused ? (uint32_t)(nbox * p.box_m * BK) : (uint32_t)kAStageBytes;
        // (CTA pair: A, B and both scale tiles on the full barrier; single CTA:
        // the scale atoms on sf_loaded, for the scale warps)
        const uint32_t ab_bytes = a_bytes + L::kBStage;
        const uint32_t sf_bytes = kSfaStageBytes + L::kSfbStage;
        const uint32_t bytes = kPair ? ab_bytes + sf_bytes : ab_bytes;
        const int b_row = item.nt * kBN + (kPair ? (int)rank * (kBN / 2) : 0);
        // One load per step first: when the copy role is ahead every segment
        // of the item's steps is already staged and the per-segment checks
        // (a round trip to L2 each) are skipped.  Only for an item without a K
        // split: it reads every segment, so no segment of the slot's next step
        // can be published (and counted) before this item has read it.
        if (pid == 0) TRACE(4, w, 0);
        bool all_staged = !fused;
        if (fused && p.step_credits) {
            // whole-step fill: wait until every segment of the item's steps is staged
            // (exact with step credits: a slot's next step is copied only after all of
            // this step's segments were read, which needs them all published first)
            int last_s = -1;
            for (int b = 0; b < nbox; ++b) {
                const int s = (mt * BM + b * p.box_m) / p.cm;
                if (s == last_s) continue;
                last_s = s;
                const unsigned long long need =
                    (unsigned long long)(s / p.bn + 1) * (unsigned long long)(p.R * p.chunks_per_seg);
                if (!wait_counter(p, ctl, p.flags + FlagLayout::staged(s % p.bn, p.bn, p.R), need, kRoleTma, s, -1,
                                  s % p.bn))
                    return;
            }
            fence_proxy_async_global();
            all_staged = true;
        } else if (fused && item.S == 1) {
            all_staged = true;
            int last_s = -1;
            for (int b = 0; b < nbox && all_staged; ++b) {
                const int s = (mt * BM + b * p.box_m) / p.cm;
                if (s == last_s) continue;
                last_s = s;
                const unsigned long long need =
                    (unsigned long long)(s / p.bn + 1) * (unsigned long long)(p.R * p.chunks_per_seg);
                all_staged = ld_acquire_u64(p.flags + FlagLayout::staged(s % p.bn, p.bn, p.R)) >= need;
            }
            if (all_staged) fence_proxy_async_global();
            if (pid == 0) TRACE(5, w, all_staged ? 1000 : 2000);
        }
        for (int i = 0; i < item.nseg; ++i) {
            const int r = item.seg_lo + (i + item.rot) % item.nseg;
            bool published = all_staged;
            for (int kb = 0; kb < p.kb_per_seg; ++kb, ++it) {
                if (it % kProducers != pid) continue;
                if (!published) {
                    for (int b = 0; b < nbox; ++b) {
                        const int row0 = mt * BM + b * p.box_m;
                        const int s = row0 / p.cm;
                        const int slot = s % p.bn;
                        const unsigned long long target =
                            (unsigned long long)(s / p.bn + 1) * (unsigned long long)p.chunks_per_seg;
                        if (!wait_counter(p, ctl, p.flags + FlagLayout::filled(slot, r, p.R), target, kRoleTma, s,
                                          r, slot))
                            return;
                    }
                    fence_proxy_async_global();   // the ring was written through the generic proxy
                    published = true;
                    TRACE(5, w, r);
                }
                const int stage = it % L::kStg;
                const uint32_t ph = (uint32_t)(it / L::kStg) & 1u;
                // (CTA pair: empty is completed by the even CTA's MMA commit)
                if (!wait_mbar(p, ctl, &ctl->empty[stage], ph ^ 1u, kRoleTma, kPair)) return;
                uint64_t* bar = &ctl->full[stage];
                const int kx = kb * BK;
                const int kg = r * p.ka + kx;
                uint8_t* a_dst = sA + (size_t)stage * kAStageBytes;
                if (kPair) {
                    // A rows of this CTA's m-tile, its half of the tile's B rows,
                    // its rows' A scale atom and the B scale atoms of all 256
                    // columns.  The even CTA arms the stage for both CTAs' bytes; the
                    // odd CTA only issues (a remote arrive per stage would hold its
                    // producer for a round trip).  Completions that land before the
                    // arm leave the transaction count negative; the phase completes
                    // only after the arrival.
                    const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    ctl->tx_own[stage] = bytes;
                    if (rank == 0) {
                        const int mt_odd = cta_mtile<kPair>(item, 1);
                        const uint32_t odd_a = fused ? (uint32_t)(num_boxes(p, mt_odd) * p.box_m * BK)
                                                     : (uint32_t)kAStageBytes;
                        const uint32_t odd = odd_a + L::kBStage + sf_bytes;
                        ctl->tx_odd[stage] = odd;
                        mbar_arrive_expect_tx(bar, bytes + odd);
                    }
                    if (fused) {
                        for (int b = 0; b < nbox; ++b) {
                            const int row0 = mt * BM + b * p.box_m;
                            const int s = row0 / p.cm;
                            const int ring_row = ((s % p.bn) * p.R + r) * p.cm + (row0 - s * p.cm);
                            tma_load_2d_pair(a_dst + (size_t)b * p.box_m * BK, tma, fb, kx, ring_row, pol_stream);
                        }
                    } else {
                        tma_load_2d_pair(a_dst, tma, fb, kg, mt * BM, pol_stream);
                    }
                    tma_load_2d_pair(sB + (size_t)stage * L::kBStage, tmb, fb, kg, b_row, pol_keep);
                    const int kbg = kg / BK;
                    tma_load_2d_pair(sSfa + (size_t)stage * kSfaStageBytes, tm_sfa, fb, 0,
                                     2 * (kbg * p.Mg + mt), pol_stream);
                    tma_load_2d_pair(sSfb + (size_t)stage * L::kSfbStage, tm_sfb, fb, 0,
                                     2 * (kbg * p.Ng2 + item.nt * L::kSfbAtoms), pol_keep);
                    ctl->issued[pid] = it + 1;
                    TRACE(14, it, pid);
                    continue;
                }
                // the scale atoms first, on their own barrier: the scale warps put
                // them into TMEM while A and B are still on their way
                {
                    uint64_t* sbar = &ctl->sf_loaded[stage];
                    const int kbg = kg / BK;
                    mbar_arrive_expect_tx(sbar, sf_bytes);
                    bulk_load(sSfa + (size_t)stage * kSfaStageBytes, p.sfa + ((size_t)kbg * p.Mg + mt) * kSfAtomBytes,
                              kSfaStageBytes, sbar);
                    // the scales of all the tile's columns
                    bulk_load(sSfb + (size_t)stage * L::kSfbStage,
                              p.sfb + ((size_t)kbg * p.Ng2 + (size_t)item.nt * L::kSfbAtoms) * kSfAtomBytes,
                              L::kSfbStage, sbar);
                }
                mbar_arrive_expect_tx(bar, bytes);
                if (fused) {
                    for (int b = 0; b < nbox; ++b) {
                        const int row0 = mt * BM + b * p.box_m;
                        const int s = row0 / p.cm;
                        const int ring_row = ((s % p.bn) * p.R + r) * p.cm + (row0 - s * p.cm);
                        tma_load_2d_hint(a_dst + (size_t)b * p.box_m * BK, tma, bar, kx, ring_row, pol_stream);
                    }
                } else if (p.direct) {
                    // the A tile straight from segment r (no exchange, no pack); all-gather:
                    // from the input block holding the tile (seg_rows is a multiple of BM)
                    const SegRow src = seg_row(p, r, mt * BM);
                    tma_load_2d_hint(a_dst, p.seg_maps + src.seg, bar, seg_col0(p, r) + kx, src.row, pol_stream);
                } else {
                    tma_load_2d_hint(a_dst, tma, bar, kg, mt * BM, pol_stream);
                }
                tma_load_2d_hint(sB + (size_t)stage * L::kBStage, tmb, bar, kg, b_row, pol_keep);
                ctl->issued[pid] = it + 1;
                TRACE(14, it, pid);
            }
        }
    }
}

// Return the credit of segment r of the staging steps an m-tile's rows came from.
__device__ __forceinline__ void return_segment_credit(const GemmParams& p, int mt, int r) {
    const int nbox = num_boxes(p, mt);
    int last_s = -1;
    for (int b = 0; b < nbox; ++b) {
        const int s = (mt * BM + b * p.box_m) / p.cm;
        if (s != last_s) {
            red_relaxed_add_u64(p.flags + FlagLayout::drained(s % p.bn, r, p.bn, p.R), 1ull);
            last_s = s;
        }
    }
}

// The credit helper (fused kernel, warp 13, one lane; in a CTA pair the even
// CTA's, for both m-tiles): walks the (item, segment) sequence of the MMA
// thread and returns each segment's credit once the MMA thread has passed the
// full barrier of the segment's last K block (ctl->consumed counts the stages
// it passed), i.e. once every TMA read of the segment has landed in shared
// memory.  The copy workers that wait for the credit then overwrite ring slots
// whose reads have completed.  It polls rarely: a credit that arrives a
// microsecond late costs nothing while the ring is ahead.
template <bool kPair>
__device__ void credit_role(const GemmParams& p, SmemCtl* ctl) {
    int start = 0;   // stages of the items before this one
    for (int w = first_item<kPair>(); w < p.W; w += item_stride<kPair>()) {
        const Item item = decode_item(p, w);
        for (int i = 0; i < item.nseg; ++i) {
            const int need = start + (i + 1) * p.kb_per_seg;   // stages passed once segment i has landed
            if (ctl->consumed < need) {
                const uint64_t t0 = globaltimer();
                for (uint32_t n = 1; ctl->consumed < need; ++n) {
                    if (ctl->abort) return;
                    __nanosleep(512);
                    if ((n & 15) == 0 && globaltimer() - t0 > (uint64_t)p.timeout_ns) {
                        record_error(p, kErrTimeout, kRoleMma, -1, i, -1, (long long)ctl->consumed, need);
                        ctl->abort = 1;
                        return;
                    }
                }
            }
            const int r = item.seg_lo + (i + item.rot) % item.nseg;
            return_segment_credit(p, cta_mtile<kPair>(item, 0), r);
            if (kPair) return_segment_credit(p, cta_mtile<kPair>(item, 1), r);
        }
        start += item.nseg * p.kb_per_seg;
    }
}

// Scale factors to TMEM, per stage, into the stage's own TMEM scale columns.
// CTA pair: the MMA thread copies them from the stage (tcgen05.cp
// 32x128b.warpx4: a 512-byte atom lands in 4 TMEM columns, the same 32 x 16
// bytes in every lane quarter; each CTA copies its own shared memory into its
// own TMEM).  Single CTA: the scale warps write the same columns with
// tcgen05.st from the stage as soon as its scale atoms have landed, ahead of
// A and B (measured on GB300: the copies in the MMA issue stream cost about
// a fifth of the MMA rate, the stores by other warps do not).
template <bool kPair, int kBN>
__device__ void mma_role(const GemmParams& p, uint32_t tmem, uint8_t* sA, uint8_t* sB, uint8_t* sSfa,
                         uint8_t* sSfb, SmemCtl* ctl, bool fused) {
    using L = Lay<kPair, kBN>;
    // Instruction descriptor, kind::mxf8f6f4 with block scaling: A / B element
    // types at [7,10) / [10,13) (E4M3 0, E5M2 1), both K-major, N>>3 at
    // [17,23), scale type UE8M0 at bit 23, M>>4 at [24,29) (M = 256 for a CTA
    // pair); B/A scale-factor byte ids at [4,6) and [29,31) select which of the
    // four 32-wide K blocks held in each 32-bit TMEM scale column is used.
    constexpr uint32_t kM = kPair ? 2 * BM : BM;
    const uint32_t idesc_base = ((uint32_t)p.fmt_a << 7) | ((uint32_t)p.fmt_b << 10) |
                                ((uint32_t)(kBN >> 3) << 17) | (1u << 23) | ((kM >> 4) << 24);
    int it = 0;
    int n = 0;   // items done; item n accumulates in buffer n % kAccBufs
    for (int w = first_item<kPair>(); w < p.W; w += item_stride<kPair>(), ++n) {
        const Item item = decode_item(p, w);
        const int buf = n % L::kAccBufs;
        const uint32_t acc_ph = (uint32_t)(n / L::kAccBufs) & 1u;
        const uint32_t acc_col = tmem + kTmemAccCol + (uint32_t)(buf * kBN);
        // (CTA pair: acc_empty counts the epilogue warps of both CTAs)
        if (!wait_mbar(p, ctl, &ctl->acc_empty[buf], acc_ph ^ 1u, kRoleMma, kPair)) return;
        tc_fence_after();
        TRACE(1, w, 0);
        const int total = item.nseg * p.kb_per_seg;
        for (int j = 0; j < total; ++j) {
            const int stage = it % L::kStg;
            const uint32_t ph = (uint32_t)(it / L::kStg) & 1u;
            TRACE(15, it, 0);
            // (CTA pair: full covers both CTAs' loads of the stage, scales included)
            if (!wait_mbar(p, ctl, &ctl->full[stage], ph, kRoleMma, kPair)) return;
            TRACE(11, it, 0);
            ctl->consumed = it + 1;
            if (!kPair && !wait_mbar(p, ctl, &ctl->sf_ready[stage], ph, kRoleMma)) return;
            if (j == 0) TRACE(2, w, 0);
            tc_fence_after();
            const uint32_t sf_t = tmem + kTmemSfCol + (uint32_t)stage * L::kSfCols;
            const uint64_t adesc = smem_desc(smem_u32(sA + (size_t)stage * kAStageBytes), 16, 1024, kLayoutSw128);
            const uint64_t bdesc = smem_desc(smem_u32(sB + (size_t)stage * L::kBStage), 16, 1024, kLayoutSw128);
            if (kPair) {
                const uint32_t sfa_s = smem_u32(sSfa + (size_t)stage * kSfaStageBytes);
                const uint32_t sfb_s = smem_u32(sSfb + (size_t)stage * L::kSfbStage);
                tc_cp_32x128b_warpx4_pair(sf_t, smem_desc(sfa_s, 0, 128, kLayoutNone));
#pragma unroll
                for (int a = 0; a < L::kSfbAtoms; ++a)
                    tc_cp_32x128b_warpx4_pair(sf_t + 4 + 4 * a, smem_desc(sfb_s + a * kSfAtomBytes, 0, 128, kLayoutNone));
#pragma unroll
                for (int k = 0; k < BK / 32; ++k) {
                    const uint32_t idesc = idesc_base | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                    mma_mxf8f6f4_pair(acc_col, adesc + 2ull * k, bdesc + 2ull * k, idesc, sf_t, sf_t + 4, (j | k) != 0);
                }
                tc_commit_pair_multicast(&ctl->empty[stage], 0x3);
            } else {
#pragma unroll
                for (int k = 0; k < BK / 32; ++k) {
                    const uint32_t idesc = idesc_base | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                    // +32 bytes along K inside the 128-byte swizzle atom = +2 in the encoded start address
                    mma_mxf8f6f4(acc_col, adesc + 2ull * k, bdesc + 2ull * k, idesc, sf_t, sf_t + 4, (j | k) != 0);
                }
                tc_commit(&ctl->empty[stage]);
            }
            TRACE(16, it, 0);
            ++it;
            // (the staging credits of the segments whose loads this thread saw
            // land, ctl->consumed, are returned by the credit helper: any extra
            // work per segment here, even a shared-memory store, measured
            // 45-80 us slower on the 8192^3 workload on GB300, and a global
            // atomic a fifth of the kernel's time)
        }
        if (kPair)
            tc_commit_pair_multicast(&ctl->acc_full[buf], 0x3);
        else
            tc_commit(&ctl->acc_full[buf]);
        TRACE(3, w, 0);
    }
}

// The scale warps of the single-CTA kernel (epilogue warps 6..9, one per lane
// quarter): for stages sf_it .. upto-1, as soon as a stage's scale atoms have
// landed, this warp writes its 32 TMEM lanes of the stage's scale columns
// with what the tcgen05.cp form would replicate there (lane l, column c of an
// atom's 4 columns = the atom's 32-bit word l*4 + c), then arrives on
// sf_ready[stage] (count 4).  A stage's columns are free again once its
// scales landed anew: the producer reloads a stage only after the MMAs that
// read it completed.
template <bool kPair, int kBN>
__device__ bool store_scales(const GemmParams& p, SmemCtl* ctl, uint32_t tmem, const uint8_t* sSfa,
                             const uint8_t* sSfb, int& sf_it, int upto, int lane, int quarter) {
    using L = Lay<kPair, kBN>;
    for (; sf_it < upto; ++sf_it) {
        const int stage = sf_it % L::kStg;
        const uint32_t ph = (uint32_t)(sf_it / L::kStg) & 1u;
        if (!wait_mbar_warp(p, ctl, &ctl->sf_loaded[stage], ph, kRoleEpi)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + kTmemSfCol + (uint32_t)stage * L::kSfCols;
        const uint4 va = reinterpret_cast<const uint4*>(sSfa + (size_t)stage * kSfaStageBytes)[lane];
        tmem_st_32x32b_x4(taddr, va);
#pragma unroll
        for (int a = 0; a < L::kSfbAtoms; ++a) {
            const uint4 vb =
                reinterpret_cast<const uint4*>(sSfb + (size_t)stage * L::kSfbStage + (size_t)a * kSfAtomBytes)[lane];
            tmem_st_32x32b_x4(taddr + 4 + 4 * a, vb);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->sf_ready[stage]);
    }
    return true;
}

// This thread has read its share of accumulator buffer `buf` (its tcgen05.ld
// completed): release the buffer for a later item.  Single CTA: every
// epilogue thread arrives (count kEpiThreads).  CTA pair: one arrival per
// epilogue warp of either CTA, on the even CTA's barrier (count 2 * kEpiWarps;
// the warps arrive independently, so no warp of a CTA that gives up early can
// hold the others).
template <bool kPair>
__device__ __forceinline__ void release_accumulator(SmemCtl* ctl, int buf, int lane, uint32_t rank) {
    tc_fence_before();
    if (kPair) {
        __syncwarp();
        if (lane == 0) {
            if (rank == 0)
                mbar_arrive(&ctl->acc_empty[buf]);
            else
                mbar_arrive_remote(mapa_shared(smem_u32(&ctl->acc_empty[buf]), 0));
        }
    } else {
        mbar_arrive(&ctl->acc_empty[buf]);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Store one 32-row x 32-column BF16 chunk of C: this warp's 32 rows (one per
// lane, 16 packed words each) go to the warp's shared staging buffer as
// 64-byte rows in the 64-byte swizzle (16-byte unit j of row r at unit
// j ^ ((r >> 1) & 3), conflict-free for the 32 lanes), then lane 0 stores the
// box with TMA at column x, row y; rows past M and columns past N are not
// written.  Lane 0 owns the bulk group: before the buffer is rewritten its
// previous store must have finished reading it.
__device__ __forceinline__ void store_c_chunk(const GemmParams& p, const CUtensorMap* tmc, uint8_t* buf, int lane,
                                              const uint32_t* w, int x, int y, int ylim) {
    if (lane == 0 && !p.c_host) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int pj = j ^ ((lane >> 1) & 3);
        *reinterpret_cast<uint4*>(buf + lane * 64 + pj * 16) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
    if (p.c_host) {
        // C in a host buffer: generic 16-byte stores from the staging buffer, four
        // lanes per 64-byte row segment (8 rows per warp store); they stream over
        // the host link while the next items run.  Units of 8 columns are all
        // inside N or all past it (N % 16 == 0).
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int u = k * 32 + lane, r = u >> 2, c = u & 3;
            const int gx = x + c * 8;
            if (y + r < ylim && gx < p.N)
                *reinterpret_cast<uint4*>(p.c_host + (size_t)(y + r) * p.N + gx) =
                    *reinterpret_cast<const uint4*>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) * 16));
        }
        __syncwarp();   // (read out before the next chunk rewrites the buffer)
        return;
    }
    fence_proxy_async_shared();   // the generic-proxy writes, before the TMA (async proxy) reads them
    __syncwarp();
    if (lane == 0 && x < p.N && y < ylim) {
        tma_store_2d_hint(tmc, buf, x, y, l2_policy_evict_first());   // C is written once: do not keep it in L2
        bulk_commit_group();
    }
}

// fp32 sum of 8 BF16 values (one 16-byte vector, column order) into acc
__device__ __forceinline__ void add_bf16x8(float* acc, const uint4& t) {
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        acc[2 * e] += __uint_as_float(w[e] << 16);
        acc[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
    }
}

__device__ __forceinline__ void wait_value_u64(const GemmParams& p, SmemCtl* ctl, const unsigned long long* ptr,
                                               unsigned long long want, bool* ok) {
    // like wait_counter, for an exact epoch value
    if (!wait_counter(p, ctl, ptr, want, kRoleEpi, -1, -1, -1)) *ok = false;
}

template <int kBN>
__device__ bool split_reduce(const GemmParams& p, SmemCtl* ctl, const CUtensorMap* tmc, uint8_t* cbuf, int ep,
                             int lane, const Item& item, int mt, int w);

template <bool kFused, bool kPair, int kBN>
__device__ void epilogue_role(const GemmParams& p, uint32_t tmem, SmemCtl* ctl, int warp, int lane, uint32_t rank,
                              const CUtensorMap* tmc, uint8_t* sEpi, const uint8_t* sSfa, const uint8_t* sSfb) {
    using L = Lay<kPair, kBN>;
    const int ep = warp - kWarpEpi0;         // 0..7
    const int quarter = warp & 3;            // TMEM lanes this warp may access: 32*quarter .. +31
    const int half = ep >> 2;                // accumulator columns (kBN/2)*half .. +kBN/2-1
    const bool leader = (ep == 0 && lane == 0);
    // Single-CTA kernel: warps 6..9 (one per lane quarter) are also the scale
    // warps.  Before they drain item n's accumulator they write the scales of
    // its stages and of the next item's first ones, up to kStg stages past
    // item n (the producer can load those once item n's MMAs are done) and not
    // past the next item (on the fused path a later item's rows may wait for
    // staging credits that the next item returns).
    const bool sf_warp = !kPair && warp >= kWarpSf0 && warp < kWarpSf0 + kSfWarps;
    bool sf_ok = true;
    int sf_it = 0;      // next stage whose scales this warp writes
    int item_end = 0;   // stages of the items up to and including the current one
    const bool together = p.S > 1 || p.S_tail > 1;   // the launch has split items
    bool dead = false;                                // (then) this warp gave up on a whole-tile item
    int n = 0;   // items done; item n is in accumulator buffer n % kAccBufs
    for (int w = first_item<kPair>(); w < p.W; w += item_stride<kPair>(), ++n) {
        const Item item = decode_item(p, w);
        const int mt = cta_mtile<kPair>(item, rank);
        const int buf = n % L::kAccBufs;
        const uint32_t acc_ph = (uint32_t)(n / L::kAccBufs) & 1u;
        item_end += item.nseg * p.kb_per_seg;
        if (sf_warp && sf_ok && !dead) {
            int upto = item_end;
            if (w + item_stride<kPair>() < p.W) {
                const Item nx = decode_item(p, w + item_stride<kPair>());
                upto = min(item_end + L::kStg, item_end + nx.nseg * p.kb_per_seg);
            }
            sf_ok = store_scales<kPair, kBN>(p, ctl, tmem, sSfa, sSfb, sf_it, upto, lane, quarter);
        }
        // (a warp whose scale stores gave up leaves through the same path as a
        // warp whose wait ran out, so the split path's named barriers see it)
        const bool got = !dead && sf_ok && wait_mbar_warp(p, ctl, &ctl->acc_full[buf], acc_ph, kRoleEpi, kPair);
        if (item.S > 1) {
            // the split path synchronises the 8 epilogue warps on named barriers:
            // leave only all together
            if (!named_barrier_and(2, kEpiThreads, got)) return;
        } else if (!got) {
            // A warp gives up alone, except in a launch with split items: there it
            // stays in the loop doing nothing, so that the next split item's vote
            // (which it joins) makes all the warps leave together.
            if (!together) return;
            dead = true;
            continue;
        }
        if (leader) TRACE(6, w, 0);
        tc_fence_after();
        const int lrow = quarter * 32 + lane;            // row inside the tile
        const int row = mt * BM + lrow;
        const int tcol = half * (kBN / 2);               // first accumulator column of this warp
        const int col0 = item.nt * kBN + tcol;
        const uint32_t tbase =
            tmem + kTmemAccCol + (uint32_t)(buf * kBN) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)tcol;
        constexpr int kChunks = kBN / 2 / 32;            // chunks of 32 columns per warp
        uint8_t* cbuf = sEpi + (size_t)ep * kEpiBufBytes;
        const int row_w = mt * BM + quarter * 32;       // first row of this warp's 32 (M % 64 == 0: all
                                                        // 32 rows are inside M or all past it)
        if (item.S == 1) {
            uint32_t packed[kBN / 4];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
                tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) packed[c * 16 + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
            }
            release_accumulator<kPair>(ctl, buf, lane, rank);   // this accumulator may now take a later item
            if (leader) TRACE(7, w, 0);
            // C; or (GEMM + ReduceScatter) block j of the rows (rs_rows, a multiple of 64,
            // so one block holds the warp's 32) to peer j's send buffer, this rank's
            // block to out; rows past M are not stored
            const CUtensorMap* dst = tmc;
            int y = row_w, ylim = p.M;
            const bool rs = !kFused && p.rs_rows > 0;   // (the staging kernel never reduce-scatters)
            if (rs) {
                const int blk = row_w < p.M ? row_w / p.rs_rows : -1;
                dst = (blk >= 0 && (blk != p.rs_own || p.rs_publish)) ? p.send_maps + blk : tmc;
                y = blk >= 0 ? row_w - blk * p.rs_rows : 0;
                ylim = blk >= 0 ? p.rs_rows : 0;
            }
            if (p.c_host && !rs) {
                // C in a host buffer: the warp's rows go through the staging buffer
                // kHostRows at a time (a lane writes its row's kHostCols columns), so
                // that every warp store writes whole row pieces of 2 * kHostCols bytes.
                // Measured on GB300 over the host link (8192^3): 64-byte pieces
                // 145 GB/s, 128 and 256 bytes 163 GB/s, a thread per row 3.5x slower.
                constexpr int kHostCols = kBN / 2;                                 // columns per round
                constexpr int kUnits = kHostCols / 8;                              // 16-byte units per row
                constexpr int kHostRows = kEpiBufBytes / (2 * kHostCols);          // rows per round
#pragma unroll
                for (int c = 0; c < kBN / 2; c += kHostCols) {
#pragma unroll
                    for (int h = 0; h < 32 / kHostRows; ++h) {
                        if (lane / kHostRows == h) {
                            const int rr = lane % kHostRows;
#pragma unroll
                            for (int u = 0; u < kUnits; ++u)
                                *reinterpret_cast<uint4*>(cbuf + rr * (kUnits * 16) + ((u ^ (rr & 7)) * 16)) =
                                    make_uint4(packed[c / 2 + 4 * u], packed[c / 2 + 4 * u + 1],
                                               packed[c / 2 + 4 * u + 2], packed[c / 2 + 4 * u + 3]);
                        }
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < kHostRows * kUnits / 32; ++k) {
                            const int t = k * 32 + lane, rr = t / kUnits, u = t % kUnits;
                            const int gy = row_w + h * kHostRows + rr, gx = col0 + c + u * 8;
                            if (gy < p.M && gx < p.N)
                                *reinterpret_cast<uint4*>(p.c_host + (size_t)gy * p.N + gx) =
                                    *reinterpret_cast<const uint4*>(cbuf + rr * (kUnits * 16) + ((u ^ (rr & 7)) * 16));
                        }
                        __syncwarp();   // (read out before the next round rewrites the buffer)
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    store_c_chunk(p, dst, cbuf, lane, packed + c * 16, col0 + c * 32, y, ylim);
            }
            if (rs && mt * BM < (p.rs_own + 1) * p.rs_rows && (mt + 1) * BM > p.rs_own * p.rs_rows) {
                // a tile with rows of this rank's block: once this warp's stores have
                // landed, count it for the copy warps that sum those rows
                if (lane == 0) {
                    bulk_wait_all();
                    fence_proxy_async_global();
                    fence_acq_rel_gpu();
                    red_relaxed_add_u64(p.rs_cnt + (size_t)mt * p.Nt + item.nt, 1ull);
                }
                __syncwarp();
            }
        } else {
            // Every split writes its fp32 partial, frees the accumulator (so the next
            // item's MMAs overlap) and publishes ready[tile][q].  Partial tile layout
            // [kBN/4][BM][4]: thread `lrow` of a warp stores the float4 of columns
            // 4g..4g+3 at (g*BM + lrow)*4, so each warp store covers 512 contiguous bytes.
            const size_t slot = split_slot(p, item, mt);
            float* dst = p.partial + (slot * item.S + item.q) * (size_t)(BM * kBN) + ((size_t)(tcol / 4) * BM + lrow) * 4;
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
                tc_wait_ld();
                if (row < p.M) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(dst + (size_t)(c * 8 + j) * BM * 4) =
                            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            }
            release_accumulator<kPair>(ctl, buf, lane, rank);
            __threadfence();
            named_barrier_sync(2, kEpiThreads);
            if (leader) {
                asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.ready + slot * item.S + item.q),
                             "l"(p.launch_id)
                             : "memory");
                TRACE(30, w, item.q);
            }
            if (!split_reduce<kBN>(p, ctl, tmc, cbuf, ep, lane, item, mt, w)) return;
        }
    }
}

// The split-K sums of item (tile, q), right after this split has published
// its partial (the MMA thread meanwhile runs the next item): wait until every
// split of the tile has published, then sum this split's share of the tile,
// the units of 32 rows x 32 columns inside M numbered q, q + S, q + 2S, ...,
// spread over the 8 epilogue warps (M is a multiple of 64, so a 32-row group
// is all inside M or all past it).  Each unit sums the S partials in the
// fixed order q = 0..S-1, the next split's loads in flight while the previous
// one is added, and stores its BF16 32 x 32 box of C.  Every wait ends: the
// K split is the innermost item index, so a tile's splits are consecutive
// items, and with no more splits than CTAs the persistent grid runs them on
// different CTAs in one round or two adjacent ones; by induction over the
// rounds every CTA reaches and publishes each of its items (all CTAs are
// resident).  False when the wait gave up.
template <int kBN>
__device__ bool split_reduce(const GemmParams& p, SmemCtl* ctl, const CUtensorMap* tmc, uint8_t* cbuf, int ep,
                             int lane, const Item& item, int mt, int w) {
    const bool leader = (ep == 0 && lane == 0);
    const int S = item.S;
    const size_t slot = split_slot(p, item, mt);
    bool ok = true;
    if (leader) {
        for (int q = 0; q < S && ok; ++q)
            if (q != item.q) wait_value_u64(p, ctl, p.ready + slot * S + q, p.launch_id, &ok);
        TRACE(31, w, 0);
    }
    if (!named_barrier_and(2, kEpiThreads, ok)) return false;   // the leader's outcome, for all
    const float* part_tile = p.partial + slot * (size_t)S * (BM * kBN);
    const int rows_tile = min(BM, p.M - mt * BM);
    const int units = ((rows_tile + 31) / 32) * (kBN / 32);
#pragma unroll 1
    for (int u = item.q + S * ep; u < units; u += S * kEpiWarps) {
        const int rg = u / (kBN / 32), cc = u - rg * (kBN / 32);
        const float* base = part_tile + ((size_t)(cc * 8) * BM + (size_t)(rg * 32 + lane)) * 4;
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
#pragma unroll 1
        for (int q = 0; q < S; ++q) {
            const float* src = base + (size_t)q * (BM * kBN);
            uint4 t[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) t[j] = ld_cg_v4(src + (size_t)j * BM * 4);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                acc[4 * j] += __uint_as_float(t[j].x);
                acc[4 * j + 1] += __uint_as_float(t[j].y);
                acc[4 * j + 2] += __uint_as_float(t[j].z);
                acc[4 * j + 3] += __uint_as_float(t[j].w);
            }
        }
        uint32_t wds[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            wds[j] = pack_bf16x2(__float_as_uint(acc[2 * j]), __float_as_uint(acc[2 * j + 1]));
        store_c_chunk(p, tmc, cbuf, lane, wds, item.nt * kBN + cc * 32, mt * BM + rg * 32, p.M);
    }
    if (leader) TRACE(32, w, 0);
    return true;
}

// One warp copies `bytes` (a multiple of 16): 16 loads of 16 bytes in flight
// per lane (8 KiB per round), then the stores.
__device__ __forceinline__ void copy_bytes(const uint8_t* src, uint8_t* dst, long long bytes, int lane) {
    constexpr int U = 16;
    const long long n16 = bytes >> 4;
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (long long base = lane; base < n16; base += 32LL * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = base + (long long)u * 32;
            if (i < n16) v[u] = ld_nc_v4(s + i);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = base + (long long)u * 32;
            if (i < n16) d[i] = v[u];
        }
    }
}

// One warp copies nrows rows of row_bytes (a multiple of 16) from rows
// src_ld bytes apart into consecutive rows: 8 loads of 16 bytes in flight
// per lane, then the stores.
__device__ __forceinline__ void copy_rows(const uint8_t* src, int src_ld, uint8_t* dst, int row_bytes, int nrows,
                                          int lane) {
    constexpr int U = 8;
    const int vpr = row_bytes >> 4;
    const int n16 = nrows * vpr;
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (int base = lane; base < n16; base += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * 32;
            if (i < n16) {
                const int row = i / vpr;
                v[u] = ld_nc_v4(src + (size_t)row * src_ld + (size_t)(i - row * vpr) * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * 32;
            if (i < n16) d[i] = v[u];
        }
    }
}

// GEMM + ReduceScatter, this rank's rows: the copy warps (idle otherwise in
// the kernel without staging) claim tasks of 8 rows of out x one n-tile, wait
// until the 8 epilogue warps of the tile that computed them have stored this
// rank's BF16 partial there, and replace it by the sum over ranks j = 0..R-1
// of block `rank` of rank j's partial (the stored value for j == rank,
// recv[j] otherwise): fp32 adds in that order from 0, one rounding to BF16.
__device__ void rs_reduce_role(const GemmParams& p, SmemCtl* ctl, int lane) {
    constexpr int kRows = 8, U = 4, Q = 4;   // rows per task; rows and ranks loaded at once
    const int n_tasks = (p.rs_rows / kRows) * p.Nt;
    const int vpr = p.tile_n / 8;            // 16-byte vectors in a tile row: one per lane
    unsigned long long* next = p.flags + FlagLayout::copy_next(p.bn, p.R);
    uint16_t* out = p.C;
    const uint16_t* own_src = p.rs_publish ? p.rs_pub : out;   // where this rank's partial was stored
    for (;;) {
        int t = -1;
        if (lane == 0 && !ctl->abort) {
            t = (int)atomicAdd(next, 1ull);
            if (t >= n_tasks) t = -1;
        }
        t = __shfl_sync(0xffffffffu, t, 0);
        if (t < 0) return;   // uniform over the warp
        const int g = t / p.Nt;
        const int nt = t - g * p.Nt;
        const int lr0 = g * kRows;                            // first row inside the block
        const int mt = (p.rs_own * p.rs_rows + lr0) / BM;     // the m-tile that computed them
        int ok = 1;
        if (lane == 0)
            ok = wait_counter(p, ctl, p.rs_cnt + (size_t)mt * p.Nt + nt, (unsigned long long)kEpiWarps,
                              kRoleReduce, mt, nt, -1) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
        const int col = nt * p.tile_n + lane * 8;
        if (lane < vpr && col < p.N) {   // N % 8 == 0: a vector is all inside N or all past it
#pragma unroll 1
            for (int r0 = 0; r0 < kRows; r0 += U) {
                float acc[U][8];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[u][e] = 0.0f;
                for (int q0 = 0; q0 < p.rs_R; q0 += Q) {
                    uint4 tv[U][Q];
#pragma unroll
                    for (int qq = 0; qq < Q; ++qq)
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int q = q0 + qq;
                            const size_t off = (size_t)(lr0 + r0 + u) * p.N + col;
                            tv[u][qq] = make_uint4(0u, 0u, 0u, 0u);
                            if (q == p.rs_rank)
                                tv[u][qq] = ld_cg_v4(own_src + off);
                            else if (q < p.rs_R)
                                tv[u][qq] = ld_nc_v4(p.recv[q] + off);
                        }
#pragma unroll
                    for (int qq = 0; qq < Q; ++qq)
#pragma unroll
                        for (int u = 0; u < U; ++u)
                            if (q0 + qq < p.rs_R) add_bf16x8(acc[u], tv[u][qq]);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = pack_bf16x2(__float_as_uint(acc[u][2 * e]), __float_as_uint(acc[u][2 * e + 1]));
                    *reinterpret_cast<uint4*>(out + (size_t)(lr0 + r0 + u) * p.N + col) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        __syncwarp();
    }
}

// Copy task t = (step, segment, chunk) in that order.  It may overwrite its
// ring slot once every reader of that segment of the earlier steps that used
// the slot has returned its credit.
__device__ __forceinline__ bool copy_task_ready(const GemmParams& p, int t, int per_step,
                                                unsigned long long* observed, unsigned long long* target) {
    const int s = t / per_step;
    if (s < p.bn || p.exchange_only) return true;
    const int r = (t - s * per_step) / p.chunks_per_seg;
    const int slot = s % p.bn;
    unsigned long long need = 0;
    for (int s2 = slot; s2 < s; s2 += p.bn) need += readers_of_segment(p, s2);
    if (p.step_credits) {
        // whole-step release: every segment of the slot's earlier steps read by all its readers
        unsigned long long vmin = ~0ull;
        for (int r2 = 0; r2 < p.R; ++r2) {
            const unsigned long long v2 = ld_acquire_u64(p.flags + FlagLayout::drained(slot, r2, p.bn, p.R));
            vmin = v2 < vmin ? v2 : vmin;
        }
        *observed = vmin;
        *target = need;
        return vmin >= need;
    }
    const unsigned long long v = ld_acquire_u64(p.flags + FlagLayout::drained(slot, r, p.bn, p.R));
    *observed = v;
    *target = need;
    return v >= need;
}

// The exchange of the pages (AllToAllComm::PutToAllRanks, one put per peer
// and step) becomes: for each (step, segment, chunk) in step order, wait for
// the slot's credit, copy commMSize/chunks rows of A_seg[r] into
// ring[slot][r], scatter their scales into the MMA scale layout, publish.
//
// Each copy warp of a CTA is an independent worker that claims one task at a
// time from a global counter (so a segment's chunks spread over many workers
// when its slot drains) and waits for the task's credit in place.  A task
// costs a few memory round trips of latency (claim, credit check, copy,
// publish), so the exchange keeps up by having many workers and a short
// publish: lane 0 releases the counters without waiting for a reply.
// (Measured on GB300 against holding several claimed tasks per worker and
// against claiming in pairs: both lengthen the copy of a freshly drained
// segment, which sits on the critical path of the staging ring.)
__device__ void copy_role(const GemmParams& p, SmemCtl* ctl, int lane) {
    const int per_step = p.R * p.chunks_per_seg;
    const long long chunk_bytes = (long long)p.rows_per_chunk * p.ka;
    unsigned long long* next = p.flags + FlagLayout::copy_next(p.bn, p.R);
    for (;;) {
        int chosen = -1;
        if (lane == 0 && !ctl->abort) {
            const int t = (int)atomicAdd(next, 1ull);
            if (t < p.n_copy_tasks) {
                TRACE(8, t, 0);
                unsigned long long obs = 0, tgt = 0;
                bool ok = copy_task_ready(p, t, per_step, &obs, &tgt);
                const uint64_t t0 = globaltimer();
                uint32_t nap = 64;   // back-off keeps the pollers off the counters' L2 lines
                for (uint32_t n = 1; !ok; ++n) {
                    __nanosleep(nap);
                    if (nap < 256) nap <<= 1;
                    ok = copy_task_ready(p, t, per_step, &obs, &tgt);
                    if (ok) break;
                    if (ctl->abort) break;
                    if ((n & 15) == 0) {
                        if (globaltimer() - t0 > (uint64_t)p.timeout_ns) {
                            const int s = t / per_step;
                            const int r = (t - s * per_step) / p.chunks_per_seg;
                            record_error(p, kErrTimeout, kRoleCopy, s, r, s % p.bn, (long long)obs, (long long)tgt);
                            ctl->abort = 1;
                            break;
                        }
                        if (launch_failed(p)) {
                            ctl->abort = 1;
                            break;
                        }
                    }
                }
                if (ok) {
                    chosen = t;
                    TRACE(9, t, 0);
                }
            }
        }
        const int t = __shfl_sync(0xffffffffu, chosen, 0);
        if (t < 0) return;   // uniform over the warp
        if (p.copy_skew_ns > 0 && (blockIdx.x & 3) == 0) {
            // test knob: a slow copier on every 4th CTA (a fixed delay, not a wait)
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < (uint64_t)p.copy_skew_ns) __nanosleep(256);
        }
        const int s = t / per_step;
        const int rem = t - s * per_step;
        const int r = rem / p.chunks_per_seg;
        const int c = rem - r * p.chunks_per_seg;
        const int slot = s % p.bn;
        const int row0 = s * p.cm + c * p.rows_per_chunk;
        const SegRow src = seg_row(p, r, row0);   // a chunk never straddles two input blocks
        const int ld = seg_ld(p), col0 = seg_col0(p, r);
        uint8_t* dst = p.ring + ((size_t)(slot * p.R + r) * p.cm + (size_t)c * p.rows_per_chunk) * p.ka;
        if (ld == p.ka)   // the rows of a segment are contiguous
            copy_bytes(p.A_seg[src.seg] + (size_t)src.row * p.ka, dst, chunk_bytes, lane);
        else              // all-gather: K slice r of full rows
            copy_rows(p.A_seg[src.seg] + (size_t)src.row * ld + col0, ld, dst, p.ka, p.rows_per_chunk, lane);
        // scales of these rows: one u32 (4 E8M0 bytes = one 128-K block) per
        // (row, K block), placed at (row%32)*4 + (row%128)/32 of the block's atom
        const int nsf = p.rows_per_chunk * p.kb_per_seg;
        for (int i = lane; i < nsf; i += 32) {
            const int kb = i / p.rows_per_chunk;
            const int m = row0 + (i - kb * p.rows_per_chunk);
            const uint32_t v = ld_nc_u32(p.A_sf_seg[src.seg] + (size_t)(src.row + (m - row0)) * (ld / 32) +
                                         col0 / 32 + kb * 4);
            const int kbg = r * p.kb_per_seg + kb;
            uint32_t* atom = reinterpret_cast<uint32_t*>(p.sfa_stage + ((size_t)kbg * p.Mg + m / BM) * kSfAtomBytes);
            atom[(m & 31) * 4 + ((m & 127) >> 5)] = v;
        }
        // Publish: the warp barrier orders every lane's stores before lane 0's
        // acq_rel fence (cumulative at gpu scope), which orders them before the
        // counter adds; readers acquire the counter and then read the ring
        // through the async proxy (TMA).
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0 && s != p.fault_skip_step) {
            fence_acq_rel_gpu();
            red_relaxed_add_u64(p.flags + FlagLayout::filled(slot, r, p.R), 1ull);
            red_relaxed_add_u64(p.flags + FlagLayout::staged(slot, p.bn, p.R), 1ull);
            TRACE(10, t, 0);
        }
    }
}

// This CTA's share of the B scale pack (the same byte permutation as
// pack_sfb_kernel): word (kbg, n) of the atoms = the 4 E8M0 bytes of column n
// for 128-wide K block kbg, at (n%32)*4 + (n%128)/32 of atom (kbg, n/128);
// columns past N get 0.  Tasks of 128 columns x up to kTileKb K blocks go
// round the CTAs; the nthreads threads taking part (tid, barrier sync) share
// one transposing tile in shared memory (the pipeline stages, unused yet).
template <typename Sync>
__device__ void pack_sfb_cta(const GemmParams& p, uint32_t* tile, int tid, int nthreads, Sync sync) {
    uint32_t* sfb = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(p.sfb));   // written only here
    const int kbs = p.K / BK;
    const long long tasks = atom_tile_tasks(p.Ng2, kbs);
    const uint8_t* src = p.B_scale;
    const size_t ld = (size_t)(p.K / 32);
    auto load = [&](int kbg, int n) { return ld_nc_u32(src + (size_t)n * ld + (size_t)kbg * 4); };
    for (long long t = blockIdx.x; t < tasks; t += gridDim.x) {
        const int g = (int)(t % p.Ng2), kb0 = (int)(t / p.Ng2) * kTileKb;
        pack_atom_tile(sfb, p.Ng2, p.N, g, kb0, min(kTileKb, kbs - kb0), tile, tid, nthreads, load, sync);
    }
}

// Each CTA packs the B scale atoms its own items read (see own_sfb_pack).
template <int kBN, typename Sync>
__device__ void pack_sfb_own(const GemmParams& p, uint32_t* tile, int tid, int nthreads, Sync sync) {
    uint32_t* sfb = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(p.sfb));   // written only here
    const uint8_t* src = p.B_scale;
    const size_t ld = (size_t)(p.K / 32);
    auto load = [&](int kbg, int n) { return ld_nc_u32(src + (size_t)n * ld + (size_t)kbg * 4); };
    for (int w = first_item<false>(); w < p.W; w += item_stride<false>()) {
        const Item item = decode_item(p, w);
        const int kb_lo = item.seg_lo * p.kb_per_seg, kb_hi = (item.seg_lo + item.nseg) * p.kb_per_seg;
        for (int g = item.nt * (kBN / 128); g < (item.nt + 1) * (kBN / 128); ++g)
            for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += kTileKb)
                pack_atom_tile(sfb, p.Ng2, p.N, g, kb0, min(kTileKb, kb_hi - kb0), tile, tid, nthreads, load, sync);
    }
}

// This CTA's share of the A scale pack for the direct variant (the scale part
// of pack_a_kernel): word (kbg, m) = the 4 E8M0 bytes of row m for 128-wide K
// block kbg, from segment kbg / kb_per_seg; rows past M get 0.
template <typename Sync>
__device__ void pack_sfa_cta(const GemmParams& p, uint32_t* tile, int tid, int nthreads, Sync sync) {
    uint32_t* sfa = reinterpret_cast<uint32_t*>(p.sfa_stage);
    const int kbs = p.K / BK;
    const long long tasks = atom_tile_tasks(p.Mg, kbs);
    auto load = [&](int kbg, int m) {
        const int r = kbg / p.kb_per_seg;
        const int kb = kbg - r * p.kb_per_seg;
        const SegRow src = seg_row(p, r, m);
        return ld_nc_u32(p.A_sf_seg[src.seg] + (size_t)src.row * (seg_ld(p) / 32) + seg_col0(p, r) / 32 +
                         (size_t)kb * 4);
    };
    for (long long t = blockIdx.x; t < tasks; t += gridDim.x) {
        const int g = (int)(t % p.Mg), kb0 = (int)(t / p.Mg) * kTileKb;
        pack_atom_tile(sfa, p.Mg, p.M, g, kb0, min(kTileKb, kbs - kb0), tile, tid, nthreads, load, sync);
    }
}

// ------------------------------------------------------------------ kernel
template <bool kFused, bool kPair, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    mxgemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_c,
                  const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb) {
    using L = Lay<kPair, kBN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + L::A;
    uint8_t* sB = smem + L::B;
    uint8_t* sSfa = smem + L::Sfa;
    uint8_t* sSfb = smem + L::Sfb;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + L::Ctl);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;   // 0 = the CTA that issues the MMAs

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStg; ++s) {
            mbar_init(&ctl->full[s], 1);   // (pair: the even CTA's producer arms it for both CTAs)
            mbar_init(&ctl->empty[s], 1);
        }
        for (int s = 0; s < L::kStg; ++s) {
            mbar_init(&ctl->sf_loaded[s], 1);
            mbar_init(&ctl->sf_ready[s], kSfWarps);
        }
        for (int b = 0; b < L::kAccBufs; ++b) {
            mbar_init(&ctl->acc_full[b], 1);
            mbar_init(&ctl->acc_empty[b], kPair ? 2 * kEpiWarps : kEpiThreads);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        for (int i = 0; i < kProducers; ++i) ctl->issued[i] = 0;
        ctl->consumed = 0;
#ifdef MXA2A_TRACE
        s_trace_n = 0;
#endif
        fence_mbarrier_init();
        TRACE(20, 0, 0);
    }
    if (warp == kWarpMma) {
        if (kPair) {
            tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ctl->tmem_base, kTmemCols);
            tmem_relinquish();
        }
    }
    if ((warp == kWarpTma || warp == kWarpTma1) && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_c);
        if (kPair) {
            prefetch_tensormap(&tmap_sfa);
            prefetch_tensormap(&tmap_sfb);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();   // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    if (threadIdx.x == 0) TRACE(21, 0, 0);
    if (p.sfb_inline || p.direct) {
        // every CTA packs its slice of the B scales (and, direct, of the A
        // scales); the producers wait for all of them before their first load
        // (the CTAs are co-resident)
        if (kFused) {
            // the copy warps start staging at once; the other 12 warps pack
            constexpr int kPackThreads = kThreads - kCopyWarps * 32;
            if (!is_copy_warp(warp)) {
                const int pw = warp < 10 ? warp : warp - 2;   // warps 0..9, 12, 13 -> 0..11
                auto sync = [] { named_barrier_sync(3, kPackThreads); };
                if (!kPair && own_sfb_pack(p))
                    pack_sfb_own<kBN>(p, reinterpret_cast<uint32_t*>(sA), pw * 32 + lane, kPackThreads, sync);
                else if (p.sfb_inline)
                    pack_sfb_cta(p, reinterpret_cast<uint32_t*>(sA), pw * 32 + lane, kPackThreads, sync);
                named_barrier_sync(3, kPackThreads);
                if (threadIdx.x == 0 && (kPair || !own_sfb_pack(p))) {
                    __threadfence();
                    red_release_add_u64(p.flags + FlagLayout::sfb_done(p.bn, p.R), 1ull);
                    TRACE(22, 0, 0);
                }
            }
        } else {
            auto sync = [] { __syncthreads(); };
            if (!kPair && own_sfb_pack(p))
                pack_sfb_own<kBN>(p, reinterpret_cast<uint32_t*>(sA), threadIdx.x, kThreads, sync);
            else if (p.sfb_inline)
                pack_sfb_cta(p, reinterpret_cast<uint32_t*>(sA), threadIdx.x, kThreads, sync);
            if (p.direct) pack_sfa_cta(p, reinterpret_cast<uint32_t*>(sA), threadIdx.x, kThreads, sync);
            __syncthreads();
            if (threadIdx.x == 0 && (kPair || !own_sfb_pack(p))) {
                __threadfence();
                red_release_add_u64(p.flags + FlagLayout::sfb_done(p.bn, p.R), 1ull);
                TRACE(22, 0, 0);
            }
        }
    }

    if (warp == kWarpTma || warp == kWarpTma1) {
        if (lane == 0 && !p.exchange_only)
            producer_role<kPair, kBN>(p, &tmap_a, &tmap_b, &tmap_sfa, &tmap_sfb, sA, sB, sSfa, sSfb, ctl, kFused,
                                      rank, warp == kWarpTma ? 0 : 1);
    } else if (warp == kWarpMma) {
        // (CTA pair: the even CTA issues the MMAs of both; the odd CTA's warp only owns its TMEM)
        if (lane == 0 && !p.exchange_only && rank == 0)
            mma_role<kPair, kBN>(p, tmem, sA, sB, sSfa, sSfb, ctl, kFused);
    } else if (warp < kWarpCopy0) {
        if (!p.exchange_only) {
            epilogue_role<kFused, kPair, kBN>(p, tmem, ctl, warp, lane, rank, &tmap_c, smem + L::Epi, sSfa, sSfb);
            // this warp's C stores have read its staging buffer before the CTA ends
            // (their writes are complete when the kernel is)
            if (lane == 0) bulk_wait_read_all();
        }
    } else if (kFused && warp == kWarpCredit) {
        // (CTA pair: the even CTA returns both m-tiles' credits)
        if (lane == 0 && !p.exchange_only && rank == 0) credit_role<kPair>(p, ctl);
    } else if (kFused && is_copy_warp(warp)) {
        copy_role(p, ctl, lane);
    } else if (!kFused && p.rs_rows > 0 && is_copy_warp(warp)) {
        rs_reduce_role(p, ctl, lane);
    }
    if (lane == 0) TRACE(27, warp, 0);
    __syncwarp();
    __syncthreads();
    if (threadIdx.x == 0) TRACE(24, 0, 0);

    // After an abort, let every TMA load already issued land before the CTA exits
    // (each producer waits for its own stages beyond those the MMA side consumed).
    if (!kPair && (warp == kWarpTma || warp == kWarpTma1) && lane == 0 && ctl->abort) {
        const int pid = warp == kWarpTma ? 0 : 1;
        for (int i = ctl->consumed; i < ctl->issued[pid]; ++i)
            if (i % kProducers == pid) wait_mbar_plain(p, &ctl->full[i % L::kStg], (uint32_t)(i / L::kStg) & 1u);
    }
    if (kPair) {
        // Both CTAs' producers have stopped.  Every stage past those the MMA
        // thread consumed whose loads either CTA issued completes on the even
        // CTA's full barrier.  Where the even CTA armed a stage the odd CTA never
        // loaded, the odd CTA's bytes are completed by hand; where the odd CTA
        // loaded a stage the even CTA never armed, it is armed for those bytes.
        // Then the even CTA waits until the loads have landed (a normal run has
        // no such stage).
        cluster_sync();
        if (rank == 0 && threadIdx.x == 0) {
            const uint32_t odd_issued = mapa_shared(smem_u32((const void*)&ctl->issued[0]), 1);
            const uint32_t odd_tx = mapa_shared(smem_u32((const void*)&ctl->tx_own[0]), 1);
            int iss_even[kProducers], iss_odd[kProducers], hi = 0;
            for (int q = 0; q < kProducers; ++q) {
                iss_even[q] = ctl->issued[q];
                iss_odd[q] = (int)ld_shared_cluster_u32(odd_issued + 4u * (uint32_t)q);
                hi = max(hi, max(iss_even[q], iss_odd[q]));
            }
            for (int i = ctl->consumed; i < hi; ++i) {
                const int q = i % kProducers, stage = i % L::kStg;
                const bool even = i < iss_even[q], odd = i < iss_odd[q];
                if (!even && !odd) continue;   // nothing armed, nothing in flight
                uint64_t* bar = &ctl->full[stage];
                if (even && !odd) mbar_complete_tx(bar, ctl->tx_odd[stage]);
                if (!even && odd)
                    mbar_arrive_expect_tx(bar, ld_shared_cluster_u32(odd_tx + 4u * (uint32_t)stage));
                wait_mbar_plain(p, bar, (uint32_t)(i / L::kStg) & 1u, true);
            }
        }
    }
    // All MMAs complete before TMEM is released (in a pair, the even CTA's
    // commit arrives on both CTAs' drain barriers).
    if (warp == kWarpMma && lane == 0) {
        if (kPair) {
            if (rank == 0) tc_commit_pair_multicast(&ctl->drain, 0x3);
        } else {
            tc_commit(&ctl->drain);
        }
        wait_mbar_plain(p, &ctl->drain, 0, kPair);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();   // no CTA leaves while its partner may still touch its memory
    if (warp == kWarpMma) {
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem, kTmemCols);
        else
            tmem_dealloc(tmem, kTmemCols);
        if (lane == 0) TRACE(25, 0, 0);
    }
    if ((kFused || p.sfb_inline || p.direct || (!kFused && p.rs_rows > 0)) && threadIdx.x == 0) {
        // The last CTA to finish zeroes the staging credits, the scale-pack
        // count and the reduce-scatter counts for the next launch.  The count
        // of finished CTAs releases each CTA's accesses and acquires the others'.
        unsigned long long* done = p.flags + FlagLayout::cta_done(p.bn, p.R);
        const unsigned long long prev = atom_acq_rel_add_u64(done, 1ull);
        if (prev == (unsigned long long)gridDim.x - 1) {
            // Every other CTA counted itself after its last access to these
            // words, so plain stores do (serialised atomics cost several
            // microseconds here with many segments); the next launch sees them
            // after this one's end.
            auto zero = [](unsigned long long* w) { *reinterpret_cast<volatile unsigned long long*>(w) = 0ull; };
            if (kFused) {
                zero(p.flags + FlagLayout::copy_next(p.bn, p.R));
                for (int slot = 0; slot < p.bn; ++slot) {
                    zero(p.flags + FlagLayout::staged(slot, p.bn, p.R));
                    for (int r = 0; r < p.R; ++r) {
                        zero(p.flags + FlagLayout::filled(slot, r, p.R));
                        zero(p.flags + FlagLayout::drained(slot, r, p.bn, p.R));
                    }
                }
            }
            if (p.sfb_inline || p.direct) zero(p.flags + FlagLayout::sfb_done(p.bn, p.R));
            if (!kFused && p.rs_rows > 0) {   // the reduce-scatter task counter and tile counts
                zero(p.flags + FlagLayout::copy_next(p.bn, p.R));
                for (int t = 0; t < p.Mt * p.Nt; ++t) p.rs_cnt[t] = 0ull;
            }
            zero(done);
            TRACE(26, 0, 0);
        }
    }
}

namespace {
template <bool kFused, bool kPair, int kBN>
cudaError_t prepare(int dev) {
    // the large dynamic shared memory opt-in is per device and per kernel
    static bool done[64] = {};
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&mxgemm_kernel<kFused, kPair, kBN>),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay<kPair, kBN>::Total);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

template <bool kFused, bool kPair, int kBN>
cudaError_t launch_one(const GemmParams& p, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                       const CUtensorMap& tmap_c, const CUtensorMap& tmap_sfa, const CUtensorMap& tmap_sfb, int grid,
                       cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare<kFused, kPair, kBN>(dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay<kPair, kBN>::Total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (kPair) {
        // CTA pairs of a cluster; the grid never exceeds the pairs that can be
        // resident together, which the fused kernel's credit waits rely on
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
    } else {
        // The fused kernel's CTAs wait on each other's credits, and with the
        // scale pack in the prologue every producer waits for every CTA: they
        // must all be resident at once, which a cooperative launch guarantees
        // (or refuses).
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (kPair || kFused || p.sfb_inline || p.direct) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, &mxgemm_kernel<kFused, kPair, kBN>, p, tmap_a, tmap_b, tmap_c, tmap_sfa, tmap_sfb);
}

template <bool kFused>
int max_pairs_impl() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || prepare<kFused, true, BN>(dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay<true, BN>::Total;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&mxgemm_kernel<kFused, true, BN>), &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}
}  // namespace

#ifdef MXA2A_TRACE
// Trace access for the traced build: copy out and clear.
extern "C" int mxa2a_trace_read(void* host, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(host, g_trace, bytes) != cudaSuccess) return -1;
    static unsigned char zeros[sizeof(g_trace_n)] = {};
    if (cudaMemcpyToSymbol(g_trace_n, zeros, sizeof zeros) != cudaSuccess) return -1;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_trace) != cudaSuccess || cudaMemset(ptr, 0, sizeof(g_trace)) != cudaSuccess)
        return -1;
    return kTraceCap;
}
#endif

int mxgemm_max_pairs(bool fused) { return fused ? max_pairs_impl<true>() : max_pairs_impl<false>(); }

cudaError_t launch_mxgemm(const GemmParams& p, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                          const CUtensorMap& tmap_c, int grid, bool fused, cudaStream_t stream,
                          const CUtensorMap* tmap_sf) {
    // the scale atoms' tensor maps (sfa, sfb) are read by the CTA-pair kernel only
    CUtensorMap none;
    std::memset(&none, 0, sizeof none);
    const CUtensorMap& sfa = tmap_sf ? tmap_sf[0] : none;
    const CUtensorMap& sfb = tmap_sf ? tmap_sf[1] : none;
    if (p.pair) {
        if (p.tile_n != BN || !tmap_sf) return cudaErrorInvalidValue;
        if (fused) return launch_one<true, true, BN>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
        return launch_one<false, true, BN>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
    }
    if (p.tile_n == BN_NARROW) {
        if (fused) return launch_one<true, false, BN_NARROW>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
        return launch_one<false, false, BN_NARROW>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
    }
    if (p.tile_n != BN) return cudaErrorInvalidValue;
    if (fused) return launch_one<true, false, BN>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
    return launch_one<false, false, BN>(p, tmap_a, tmap_b, tmap_c, sfa, sfb, grid, stream);
}

}  // namespace mxa2a

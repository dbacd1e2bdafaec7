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
// CTA roles (256 threads, one CTA per SM, persistent over work items):
//   warp 0   TMA producer: waits for a slot's segment to be published, then
//            streams A (from the ring, or from the packed A when unfused), B
//            and both scale tiles into a 4-stage shared-memory ring.
//   warp 1   TMEM owner and MMA issuer: copies the stage's scale factors to
//            TMEM (tcgen05.cp) and issues 4 tcgen05.mma kind::mxf8f6f4
//            block-scaled MMAs (128x256x32 each) per 128-wide K block.
//   warps 2-9 epilogue: TMEM -> registers -> BF16 -> global, or, for split
//            K, the in-kernel fixed-order reduction of the split partials.
//            Warp w drains TMEM lane quarter w%4, column half (w-2)/4.
//   warps 10-11 staging copy (fused only): copy-tasks (step, segment, chunk)
//            in step order; wait for the slot's credit, copy the rows of
//            A_seg[r] and their scales, publish.
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

#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa2a {
using namespace ptx;

struct __align__(8) SmemCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort;
    volatile int issued;     // stages issued by the TMA producer
    volatile int consumed;   // stages whose full barrier the MMA thread has passed
    volatile int copy_go;    // copy-role broadcast
    volatile int copy_task;
    volatile int ticket;     // split-K arrival order of the current tile (epilogue broadcast)
    volatile int epi_ok;     // epilogue broadcast: the other partials of the tile are ready
    volatile int epi_warp_ok[kEpiWarps];
};

constexpr size_t kSmemA = 0;
constexpr size_t kSmemB = kSmemA + (size_t)kStages * kAStageBytes;
constexpr size_t kSmemSfa = kSmemB + (size_t)kStages * kBStageBytes;
constexpr size_t kSmemSfb = kSmemSfa + (size_t)kStages * kSfaStageBytes;
constexpr size_t kSmemCtl = kSmemSfb + (size_t)kStages * kSfbStageBytes;
constexpr size_t kSmemTotal = kSmemCtl + sizeof(SmemCtl) + 1024;   // + runtime 1 KiB alignment

size_t mxgemm_smem_bytes() { return kSmemTotal; }

// ------------------------------------------------------------------ work items
struct Item {
    int mt, nt, q, seg_lo, nseg, rot;
};

// Flattened work id -> (m-tile, n-tile, K split).  Items are ordered m-tile
// major so the staging steps are consumed in order; inside an m-tile the
// n-tiles run forward on even m-tiles and backward on odd ones (zigzag), so
// consecutive m-tiles reuse the B tiles still in L2.  Each item starts its
// K loop at a rotated segment so concurrent items read different segments.
__device__ __forceinline__ Item decode_item(const GemmParams& p, int w) {
    Item it;
    const int per_m = p.Nt * p.S;
    it.mt = w / per_m;
    const int rem = w - it.mt * per_m;
    const int ntl = rem / p.S;
    it.q = rem - ntl * p.S;
    it.nt = (p.zigzag && (it.mt & 1)) ? (p.Nt - 1 - ntl) : ntl;
    it.seg_lo = it.q * p.R / p.S;
    const int seg_hi = (it.q + 1) * p.R / p.S;
    it.nseg = seg_hi - it.seg_lo;
    it.rot = p.rotate ? (it.mt + it.nt) % it.nseg : 0;
    return it;
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
__device__ bool wait_mbar(const GemmParams& p, SmemCtl* ctl, uint64_t* bar, uint32_t parity, int role) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
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
                                               int role) {
    const bool ok = wait_mbar(p, ctl, bar, parity, role);
    return __all_sync(0xffffffffu, ok);
}

// Cleanup wait: only the time limit ends it (used after an abort).
__device__ void wait_mbar_plain(const GemmParams& p, uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
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
        if (nap < 1024) nap <<= 1;
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

// ------------------------------------------------------------------ roles
__device__ void producer_role(const GemmParams& p, const CUtensorMap* tma, const CUtensorMap* tmb,
                              uint8_t* sA, uint8_t* sB, uint8_t* sSfa, uint8_t* sSfb, SmemCtl* ctl,
                              bool fused) {
    int it = 0;
    for (int w = blockIdx.x; w < p.W; w += gridDim.x) {
        const Item item = decode_item(p, w);
        const int nbox = fused ? num_boxes(p, item.mt) : 1;
        const uint32_t a_bytes = fused ? (uint32_t)(nbox * p.box_m * BK) : (uint32_t)kAStageBytes;
        const uint32_t bytes = a_bytes + kBStageBytes + kSfaStageBytes + kSfbStageBytes;
        for (int i = 0; i < item.nseg; ++i) {
            const int r = item.seg_lo + (i + item.rot) % item.nseg;
            if (fused) {
                for (int b = 0; b < nbox; ++b) {
                    const int row0 = item.mt * BM + b * p.box_m;
                    const int s = row0 / p.cm;
                    const int slot = s % p.bn;
                    const unsigned long long target =
                        (unsigned long long)(s / p.bn + 1) * (unsigned long long)p.chunks_per_seg;
                    if (!wait_counter(p, ctl, p.flags + FlagLayout::filled(slot, r, p.R), target, kRoleTma, s, r,
                                      slot))
                        return;
                }
                fence_proxy_async_global();   // the ring was written through the generic proxy
            }
            for (int kb = 0; kb < p.kb_per_seg; ++kb) {
                const int stage = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!wait_mbar(p, ctl, &ctl->empty[stage], ph ^ 1u, kRoleTma)) return;
                uint64_t* bar = &ctl->full[stage];
                mbar_arrive_expect_tx(bar, bytes);
                const int kx = kb * BK;
                const int kg = r * p.ka + kx;
                uint8_t* a_dst = sA + (size_t)stage * kAStageBytes;
                if (fused) {
                    for (int b = 0; b < nbox; ++b) {
                        const int row0 = item.mt * BM + b * p.box_m;
                        const int s = row0 / p.cm;
                        const int ring_row = ((s % p.bn) * p.R + r) * p.cm + (row0 - s * p.cm);
                        tma_load_2d(a_dst + (size_t)b * p.box_m * BK, tma, bar, kx, ring_row);
                    }
                } else {
                    tma_load_2d(a_dst, tma, bar, kg, item.mt * BM);
                }
                tma_load_2d(sB + (size_t)stage * kBStageBytes, tmb, bar, kg, item.nt * BN);
                const int kbg = kg / BK;
                bulk_load(sSfa + (size_t)stage * kSfaStageBytes,
                          p.sfa + ((size_t)kbg * p.Mg + item.mt) * kSfAtomBytes, kSfaStageBytes, bar);
                bulk_load(sSfb + (size_t)stage * kSfbStageBytes,
                          p.sfb + ((size_t)kbg * p.Ng2 + 2 * item.nt) * kSfAtomBytes, kSfbStageBytes, bar);
                ++it;
                ctl->issued = it;
            }
        }
    }
}

__device__ void mma_role(const GemmParams& p, uint32_t tmem, uint8_t* sA, uint8_t* sB, uint8_t* sSfa,
                         uint8_t* sSfb, SmemCtl* ctl, bool fused) {
    // Instruction descriptor, kind::mxf8f6f4 with block scaling: A/B E4M3 (0),
    // both K-major, N>>3 at [17,23), scale type UE8M0 at bit 23, M>>4 at
    // [24,29); B/A scale-factor byte ids at [4,6) and [29,31) select which of
    // the four 32-wide K blocks held in each 32-bit TMEM scale column is used.
    const uint32_t idesc_base = ((uint32_t)(BN >> 3) << 17) | (1u << 23) | ((uint32_t)(BM >> 4) << 24);
    int it = 0;
    uint32_t acc_ph = 0;
    for (int w = blockIdx.x; w < p.W; w += gridDim.x) {
        const Item item = decode_item(p, w);
        if (!wait_mbar(p, ctl, &ctl->acc_empty, acc_ph ^ 1u, kRoleMma)) return;
        tc_fence_after();
        const int total = item.nseg * p.kb_per_seg;
        const int nbox = fused ? num_boxes(p, item.mt) : 0;
        for (int j = 0; j < total; ++j) {
            const int stage = it % kStages;
            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
            if (!wait_mbar(p, ctl, &ctl->full[stage], ph, kRoleMma)) return;
            ctl->consumed = it + 1;
            tc_fence_after();
            const uint32_t sf_t = tmem + kTmemSfCol + (uint32_t)stage * kTmemSfColsPerStage;
            const uint32_t sfa_s = smem_u32(sSfa + (size_t)stage * kSfaStageBytes);
            const uint32_t sfb_s = smem_u32(sSfb + (size_t)stage * kSfbStageBytes);
            tc_cp_32x128b_warpx4(sf_t, smem_desc(sfa_s, 0, 128, kLayoutNone));
            tc_cp_32x128b_warpx4(sf_t + 4, smem_desc(sfb_s, 0, 128, kLayoutNone));
            tc_cp_32x128b_warpx4(sf_t + 8, smem_desc(sfb_s + kSfAtomBytes, 0, 128, kLayoutNone));
            const uint64_t adesc = smem_desc(smem_u32(sA + (size_t)stage * kAStageBytes), 16, 1024, kLayoutSw128);
            const uint64_t bdesc = smem_desc(smem_u32(sB + (size_t)stage * kBStageBytes), 16, 1024, kLayoutSw128);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
                const uint32_t idesc = idesc_base | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                // +32 bytes along K inside the 128-byte swizzle atom = +2 in the encoded start address
                mma_mxf8f6f4(tmem + kTmemAccCol, adesc + 2ull * k, bdesc + 2ull * k, idesc, sf_t, sf_t + 4,
                             (j | k) != 0);
            }
            tc_commit(&ctl->empty[stage]);
            ++it;
            if (fused && (j % p.kb_per_seg) == p.kb_per_seg - 1) {
                // Every TMA read of this segment of the ring has landed in shared
                // memory (this thread observed the stages' full barriers), so no
                // later global write can change what the MMAs read: the credit is
                // returned with a relaxed add.  A release here would make this
                // thread wait for its in-flight tensor-core work first.
                const int i = j / p.kb_per_seg;
                const int r = item.seg_lo + (i + item.rot) % item.nseg;
                int last_s = -1;
                for (int b = 0; b < nbox; ++b) {
                    const int s = (item.mt * BM + b * p.box_m) / p.cm;
                    if (s != last_s) {
                        red_relaxed_add_u64(p.flags + FlagLayout::drained(s % p.bn, r, p.bn, p.R), 1ull);
                        last_s = s;
                    }
                }
            }
        }
        tc_commit(&ctl->acc_full);
        acc_ph ^= 1u;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void wait_value_u64(const GemmParams& p, SmemCtl* ctl, const unsigned long long* ptr,
                                               unsigned long long want, bool* ok) {
    // like wait_counter, for an exact epoch value
    if (!wait_counter(p, ctl, ptr, want, kRoleEpi, -1, -1, -1)) *ok = false;
}

__device__ void epilogue_role(const GemmParams& p, uint32_t tmem, SmemCtl* ctl, int warp, int lane) {
    const int ep = warp - kWarpEpi0;         // 0..7
    const int quarter = warp & 3;            // TMEM lanes this warp may access: 32*quarter .. +31
    const int half = ep >> 2;                // accumulator columns 128*half .. +127
    const bool leader = (ep == 0 && lane == 0);
    uint32_t acc_ph = 0;
    for (int w = blockIdx.x; w < p.W; w += gridDim.x) {
        const Item item = decode_item(p, w);
        const bool got = wait_mbar_warp(p, ctl, &ctl->acc_full, acc_ph, kRoleEpi);
        if (p.S > 1) {
            // the split path synchronises the 8 epilogue warps on a named barrier:
            // leave only all together
            if (lane == 0) ctl->epi_warp_ok[ep] = got ? 1 : 0;
            named_barrier_sync(2, kEpiThreads);
            bool all = true;
#pragma unroll
            for (int e = 0; e < kEpiWarps; ++e) all = all && ctl->epi_warp_ok[e] != 0;
            if (!all) return;
        } else if (!got) {
            return;
        }
        tc_fence_after();
        const int lrow = quarter * 32 + lane;            // row inside the tile
        const int row = item.mt * BM + lrow;
        const int tcol = half * (BN / 2);                // first accumulator column of this warp
        const int col0 = item.nt * BN + tcol;
        const uint32_t tbase = tmem + kTmemAccCol + ((uint32_t)(quarter * 32) << 16) + (uint32_t)tcol;
        constexpr int kChunks = BN / 2 / 32;             // 4 chunks of 32 columns
        if (p.S == 1) {
            uint32_t packed[BN / 4];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
                tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) packed[c * 16 + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
            }
            tc_fence_before();
            mbar_arrive(&ctl->acc_empty);   // TMEM may now take the next item
            if (row < p.M) {
                uint16_t* dst = p.C + (size_t)row * p.N + col0;
#pragma unroll
                for (int j = 0; j < BN / 16; ++j) {
                    if (col0 + j * 8 < p.N)
                        *reinterpret_cast<uint4*>(dst + j * 8) =
                            make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                }
            }
        } else {
            const size_t tile = (size_t)item.mt * p.Nt + item.nt;
            if (leader) ctl->ticket = (int)atomicAdd(&p.tile_cnt[tile], 1u);
            named_barrier_sync(2, kEpiThreads);
            const bool last = ctl->ticket == p.S - 1;
            // partial tile layout [BN/4][BM][4]: thread `lrow` of a warp stores the
            // float4 of columns 4g..4g+3 at (g*BM + lrow)*4, so each warp store
            // covers 512 contiguous bytes
            float* part_tile = p.partial + tile * (size_t)p.S * (BM * BN);
            if (!last) {
                float* dst = part_tile + (size_t)item.q * (BM * BN) + ((size_t)(tcol / 4) * BM + lrow) * 4;
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
                tc_fence_before();
                mbar_arrive(&ctl->acc_empty);
                __threadfence();
                named_barrier_sync(2, kEpiThreads);
                if (leader)
                    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.ready + tile * p.S + item.q),
                                 "l"(p.launch_id)
                                 : "memory");
            } else {
                // wait until every other split of this tile has published its partial
                if (leader) {
                    bool ok = true;
                    for (int q = 0; q < p.S && ok; ++q)
                        if (q != item.q) wait_value_u64(p, ctl, p.ready + tile * p.S + q, p.launch_id, &ok);
                    ctl->epi_ok = ok ? 1 : 0;
                }
                named_barrier_sync(2, kEpiThreads);
                const bool ok = ctl->epi_ok != 0;
                uint16_t* dst = p.C + (size_t)row * p.N + col0;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
                    tc_wait_ld();
                    if (ok && row < p.M) {
                        // fixed order q = 0..S-1, whichever split finished last
                        float acc[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
                        for (int q = 0; q < p.S; ++q) {
                            if (q == item.q) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) acc[e] += __uint_as_float(v[e]);
                            } else {
                                const float* src = part_tile + (size_t)q * (BM * BN) +
                                                   ((size_t)(tcol / 4 + c * 8) * BM + lrow) * 4;
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 t = *reinterpret_cast<const float4*>(src + (size_t)j * BM * 4);
                                    acc[4 * j] += t.x;
                                    acc[4 * j + 1] += t.y;
                                    acc[4 * j + 2] += t.z;
                                    acc[4 * j + 3] += t.w;
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (col0 + c * 32 + j * 8 < p.N)
                                *reinterpret_cast<uint4*>(dst + c * 32 + j * 8) = make_uint4(
                                    pack_bf16x2(__float_as_uint(acc[8 * j]), __float_as_uint(acc[8 * j + 1])),
                                    pack_bf16x2(__float_as_uint(acc[8 * j + 2]), __float_as_uint(acc[8 * j + 3])),
                                    pack_bf16x2(__float_as_uint(acc[8 * j + 4]), __float_as_uint(acc[8 * j + 5])),
                                    pack_bf16x2(__float_as_uint(acc[8 * j + 6]), __float_as_uint(acc[8 * j + 7])));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&ctl->acc_empty);
                if (leader) p.tile_cnt[tile] = 0u;   // ready for the next launch
                if (!ok) return;
            }
        }
        acc_ph ^= 1u;
    }
}

__device__ __forceinline__ void copy_bytes(const uint8_t* src, uint8_t* dst, long long bytes, int tid) {
    constexpr int U = 8;
    const long long n16 = bytes >> 4;
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (long long base = tid; base < n16; base += (long long)kCopyThreads * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = base + (long long)u * kCopyThreads;
            if (i < n16) v[u] = ld_nc_v4(s + i);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = base + (long long)u * kCopyThreads;
            if (i < n16) d[i] = v[u];
        }
    }
}

// The exchange of the pages (AllToAllComm::PutToAllRanks, one put per peer
// and step) becomes: for each (step, segment, chunk) in step order, wait for
// the slot's credit, copy commMSize/chunks rows of A_seg[r] into
// ring[slot][r], scatter their scales into the MMA scale layout, publish.
__device__ void copy_role(const GemmParams& p, SmemCtl* ctl, int ctid) {
    const int per_step = p.R * p.chunks_per_seg;
    const long long chunk_bytes = (long long)p.rows_per_chunk * p.ka;
    const int sf_cols = p.ka / 32;
    unsigned long long* next = p.flags + FlagLayout::copy_next(p.bn, p.R);
    for (;;) {
        // Tasks are claimed from one global counter in (step, segment, chunk)
        // order, so a copy role waiting for one slot's credit never holds back
        // tasks that another CTA could already copy.
        if (ctid == 0) {
            int t = ctl->abort ? p.n_copy_tasks : (int)atomicAdd(next, 1ull);
            bool ok = t < p.n_copy_tasks;
            if (ok) {
                const int s = t / per_step;
                const int r = (t - s * per_step) / p.chunks_per_seg;
                const int slot = s % p.bn;
                if (s >= p.bn && !p.exchange_only) {
                    unsigned long long target = 0;
                    for (int s2 = slot; s2 < s; s2 += p.bn) target += readers_of_segment(p, s2);
                    ok = wait_counter(p, ctl, p.flags + FlagLayout::drained(slot, r, p.bn, p.R), target,
                                      kRoleCopy, s, r, slot);
                }
            }
            ctl->copy_task = t;
            ctl->copy_go = ok ? 1 : 0;
        }
        named_barrier_sync(1, kCopyThreads);
        if (!ctl->copy_go) return;   // uniform over the 64 copy threads
        const int t = ctl->copy_task;
        const int s = t / per_step;
        const int rem = t - s * per_step;
        const int r = rem / p.chunks_per_seg;
        const int c = rem - r * p.chunks_per_seg;
        const int slot = s % p.bn;
        const int row0 = s * p.cm + c * p.rows_per_chunk;
        copy_bytes(p.A_seg[r] + (size_t)row0 * p.ka,
                   p.ring + ((size_t)(slot * p.R + r) * p.cm + (size_t)c * p.rows_per_chunk) * p.ka, chunk_bytes,
                   ctid);
        // scales of these rows: one u32 (4 E8M0 bytes = one 128-K block) per
        // (row, K block), placed at (row%32)*4 + (row%128)/32 of the block's atom
        const int nsf = p.rows_per_chunk * p.kb_per_seg;
        for (int i = ctid; i < nsf; i += kCopyThreads) {
            const int kb = i / p.rows_per_chunk;
            const int m = row0 + (i - kb * p.rows_per_chunk);
            const uint32_t v = ld_nc_u32(p.A_sf_seg[r] + (size_t)m * sf_cols + kb * 4);
            const int kbg = r * p.kb_per_seg + kb;
            uint32_t* atom = reinterpret_cast<uint32_t*>(p.sfa_stage + ((size_t)kbg * p.Mg + m / BM) * kSfAtomBytes);
            atom[(m & 31) * 4 + ((m & 127) >> 5)] = v;
        }
        __threadfence();
        fence_proxy_async_global();
        named_barrier_sync(1, kCopyThreads);
        if (ctid == 0 && s != p.fault_skip_step)
            red_release_add_u64(p.flags + FlagLayout::filled(slot, r, p.R), 1ull);
    }
}

// ------------------------------------------------------------------ kernel
template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    mxgemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_b) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + kSmemA;
    uint8_t* sB = smem + kSmemB;
    uint8_t* sSfa = smem + kSmemSfa;
    uint8_t* sSfb = smem + kSmemSfb;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + kSmemCtl);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->acc_full, 1);
        mbar_init(&ctl->acc_empty, kEpiThreads);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->consumed = 0;
        ctl->copy_go = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kWarpTma) {
        if (lane == 0 && !p.exchange_only) producer_role(p, &tmap_a, &tmap_b, sA, sB, sSfa, sSfb, ctl, kFused);
    } else if (warp == kWarpMma) {
        if (lane == 0 && !p.exchange_only) mma_role(p, tmem, sA, sB, sSfa, sSfb, ctl, kFused);
    } else if (warp < kWarpCopy0) {
        if (!p.exchange_only) epilogue_role(p, tmem, ctl, warp, lane);
    } else if (kFused) {
        copy_role(p, ctl, threadIdx.x - kWarpCopy0 * 32);
    }
    __syncwarp();
    __syncthreads();

    // After an abort, let every TMA load already issued land before the CTA exits.
    if (warp == kWarpTma && lane == 0 && ctl->abort) {
        for (int i = ctl->consumed; i < ctl->issued; ++i)
            wait_mbar_plain(p, &ctl->full[i % kStages], (uint32_t)(i / kStages) & 1u);
    }
    // All MMAs of this CTA complete before TMEM is released.
    if (warp == kWarpMma && lane == 0) {
        tc_commit(&ctl->drain);
        wait_mbar_plain(p, &ctl->drain, 0);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if ((kFused || p.S > 1) && threadIdx.x == 0) {
        // The last CTA to finish zeroes the staging credits for the next launch,
        // and, if this launch gave up somewhere, the split-K tile counters.
        __threadfence();
        unsigned long long* done = p.flags + FlagLayout::cta_done(p.bn, p.R);
        const unsigned long long prev = atomicAdd(done, 1ull);
        if (prev == (unsigned long long)gridDim.x - 1) {
            __threadfence();
            if (kFused) {
                atomicExch(p.flags + FlagLayout::copy_next(p.bn, p.R), 0ull);
                for (int slot = 0; slot < p.bn; ++slot) {
                    for (int r = 0; r < p.R; ++r) {
                        atomicExch(p.flags + FlagLayout::filled(slot, r, p.R), 0ull);
                        atomicExch(p.flags + FlagLayout::drained(slot, r, p.bn, p.R), 0ull);
                    }
                }
            }
            if (p.S > 1 && launch_failed(p))
                for (int t = 0; t < p.Mt * p.Nt; ++t) atomicExch(&p.tile_cnt[t], 0u);
            atomicExch(done, 0ull);
            __threadfence();
        }
    }
}

cudaError_t launch_mxgemm(const GemmParams& p, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, int grid,
                          bool fused, cudaStream_t stream) {
    // the large dynamic shared memory opt-in is per device and per kernel
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* fn = fused ? reinterpret_cast<const void*>(&mxgemm_kernel<true>)
                           : reinterpret_cast<const void*>(&mxgemm_kernel<false>);
    if (dev < 0 || dev >= 64 || !attr_set[dev][fused ? 1 : 0]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTotal);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev][fused ? 1 : 0] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // The fused kernel's CTAs wait on each other's credits: they must all be
    // resident at once, which a cooperative launch guarantees (or refuses).
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = fused ? 1 : 0;
    if (fused) return cudaLaunchKernelEx(&cfg, &mxgemm_kernel<true>, p, tmap_a, tmap_b);
    return cudaLaunchKernelEx(&cfg, &mxgemm_kernel<false>, p, tmap_a, tmap_b);
}

}  // namespace mxa2a

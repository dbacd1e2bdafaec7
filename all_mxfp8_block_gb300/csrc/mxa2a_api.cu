// C ABI of libmxa2a: plan creation and validation, workspace, TMA
// descriptors, launch sequencing and status.  Host code only; the kernels
// are in mxgemm.cu and aux_kernels.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/mxa2a.h"
#include "kernels.cuh"

using namespace mxa2a;

namespace {

thread_local int g_last_error = MXA2A_OK;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D uint8 tensor [outer][inner] (inner contiguous), box [box_outer][128], 128-byte swizzle.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C: bf16 [M][N] (N contiguous), box 32 rows x 32 columns, 64-byte swizzle
// (the epilogue's TMA stores; see store_c_chunk).
bool encode_c(CUtensorMap* map, void* C, uint64_t M, uint64_t N) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {N, M};
    cuuint64_t strides[1] = {N * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Scale atoms ([blocks][512] u8) as a 2D u8 tensor of 256-byte rows (2 per
// atom), box box_rows x 256, no swizzle: the CTA-pair kernel's loads of one
// A atom (2 rows) or a tile's two B atoms (4 rows).
bool encode_atoms(CUtensorMap* map, const void* base, uint64_t atoms, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || atoms == 0) return false;
    cuuint64_t dims[2] = {256, atoms * 2};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int tile_span(int64_t M, int64_t cm, int64_t rows = BM) {
    // the most staging steps any output tile of `rows` rows touches
    int span = 1;
    const int64_t Mt = (M + rows - 1) / rows;
    for (int64_t mt = 0; mt < Mt; ++mt) {
        const int64_t r0 = mt * rows, r1 = std::min<int64_t>(M, r0 + rows) - 1;
        span = std::max<int>(span, (int)(r1 / cm - r0 / cm + 1));
    }
    return span;
}

}  // namespace

struct mxa2a_plan {
    int R;                  // K slices of the GEMM's A (1 for the all-gather)
    int64_t M, ka, N, cm;
    int bn;
    int kind = MXA2A_KIND_ALLTOALL;
    int nseg = 0;           // input buffers of A: R (all-to-all) or the ranks (all-gather)
    int64_t seg_rows = 0;   // all-gather: rows per input block; 0: all M rows
    int device = 0, sm_count = 0;
    // derived
    int64_t K = 0;
    int steps = 0, Mt = 0, Nt = 0, Mg = 0, Ng2 = 0, box_m = 128, span = 1;   // Nt: wide (256-column) tiles
    int tn_fused = BN, tn_unfused = BN;     // tile width per path (256, or 128 = the narrow tile)
    int Nt_fused = 0, Nt_unfused = 0;       // n-tiles per path
    int tile_opt = 0;                       // option: 0 automatic, 128 or 256 forced
    void* c_host = nullptr;                 // during a host-buffer run: C's host buffer (device view)
    int elem_types = 0;                     // option: element-format pair (MXA2A_OPT_ELEM_TYPES)
    int step_credits = 0;                   // option: whole-step staging credits
    int copy_skew_ns = 0;                   // test knob: delay of every 4th CTA's copies
    int S_fused = 1, S_unfused = 1, W_fused = 0, W_unfused = 0;   // K splits and work items per path
    int Wdp_fused = 0, Wdp_unfused = 0;     // items before the split tail (= W: no tail split)
    int St_fused = 1, St_unfused = 1;       // K split of the tail's tiles
    int tail_split = 1;                     // option: 1 allows the tail split
    int pair_fused = 0, pair_unfused = 0;   // CTA-pair kernel in use, per path
    int group_fused = 1, group_unfused = 1; // raster group, in m rows (tiles or tile pairs)
    int group_cap = 16;                     // option: largest unfused raster group
    int group_fused_opt = 0;                // option: fused raster group in m-tiles (0 = one)
    int allow_pair = 2;           // option: 0 never, 1 both paths, 2 automatic (the CTA-pair kernel)
    int max_pairs_fused = 0, max_pairs_unfused = 0;
    int rows_per_chunk = 1, chunks_per_seg = 1, n_copy_tasks = 0;
    int grid_fused = 0, grid_unfused = 0;
    // options
    int64_t timeout_ns = 2000000000LL;
    int force_split = 0, zigzag = 1, rotate = 0, record_events = 0, exchange_only = 0;
    int fault_skip_step = -1, grid_cap = 0;
    int64_t chunk_bytes = 0;            // option: staging copy chunk, 0 = automatic
    // workspace
    uint8_t* ws = nullptr;
    size_t ws_bytes = 0;
    uint8_t *ring = nullptr, *sfa = nullptr, *sfb = nullptr, *a_packed = nullptr;
    // split-K scratch, own allocation sized for the current splits:
    // fp32 partial tiles [Mt*Nt][S][128][256] | tile counters u32 [Mt*Nt] | ready u64 [Mt*Nt][S]
    uint8_t* split_ws = nullptr;
    float* partial = nullptr;
    unsigned long long* ready = nullptr;
    unsigned long long* flags = nullptr;
    DevStatus* status = nullptr;
    size_t ring_bytes = 0, sfa_bytes = 0, sfb_bytes = 0, apacked_bytes = 0, partial_bytes = 0, flags_bytes = 0;
    CUtensorMap tmap_ring, tmap_apacked, tmap_b, tmap_b_half;
    CUtensorMap tmap_sf[2];                 // the scale atoms in the workspace (CTA-pair kernel's loads)
    const void* tmap_b_ptr = nullptr;
    CUtensorMap tmap_c;                     // for the C pointer of the last run
    const void* tmap_c_ptr = nullptr;
    // direct variant: one tensor map per segment, in the workspace (device)
    CUtensorMap* seg_maps_dev = nullptr;
    CUtensorMap seg_maps_host[kMaxSegments];
    const void* seg_ptrs[kMaxSegments] = {};
    unsigned long long launch_id = 0, checked_launch = 0;
    // ring of (start, end) events around the main GEMM kernel of the last runs
    static constexpr int kEvRing = 4096;
    cudaEvent_t* ev0 = nullptr;
    cudaEvent_t* ev1 = nullptr;
    int ev_count = 0;       // events created
    long long ev_recorded = 0;   // runs recorded since the option was set
    int last_launches = 0;
    // host-buffer path
    uint8_t* io = nullptr;
    size_t io_bytes = 0;
    // GEMM + ReduceScatter: this rank, the ranks, rows per block
    int rs_rank = 0, rs_R = 0;
    int64_t rs_rows = 0;
    // blocks of rs_rows rows, the one summed here, and whether its partial is
    // published (GEMM + AllReduce: one block of all rows, published)
    int rs_nblk = 0, rs_own = 0, rs_publish = 0;
    uint16_t* rs_scratch = nullptr;         // the unfused path's partial P [M][N] (allocated on first use)
    CUtensorMap* send_maps_dev = nullptr;   // workspace, after the segment maps
    CUtensorMap send_maps_host[kMaxSegments];
    const void* send_ptrs[kMaxSegments] = {};
    CUtensorMap tmap_out;                   // out [rs_rows][N] of the last fused run
    const void* tmap_out_ptr = nullptr;
    unsigned long long* rs_cnt = nullptr;   // workspace: per-tile epilogue counts [Mt * 2 Nt]
    size_t rs_cnt_bytes = 0;
};

namespace mxa2a {
// aux_kernels.cu: several copies by the SMs in one launch
cudaError_t launch_copy_list(int n, const void* const* src, void* const* dst, const size_t* bytes,
                             cudaStream_t stream);
}  // namespace mxa2a

namespace {

void derive(mxa2a_plan* p) {
    p->K = (int64_t)p->R * p->ka;
    p->steps = (int)(p->M / p->cm);
    p->Mt = (int)((p->M + BM - 1) / BM);
    p->Nt = (int)((p->N + BN - 1) / BN);
    p->Mg = p->Mt;
    p->Ng2 = 2 * p->Nt;
    p->box_m = (p->cm % BM == 0) ? BM : 64;
    p->span = tile_span(p->M, p->cm);
    // K split: enough work items to fill the GPU.  The fused path can only
    // work on the output tiles whose rows sit in the staging ring at once
    // (buffer_num * commMSize rows), the unfused path on all tiles.
    // Split only when the tiles fill at most a quarter of the GPU: the in-kernel
    // reduction of the partials costs more than a partly idle GPU otherwise.
    // No more splits than persistent CTAs (CTA pairs): a tile's splits must
    // run on different ones (each waits for the others).
    const int cta_cap = p->grid_cap > 0 ? std::min(p->sm_count, p->grid_cap) : p->sm_count;
    auto split_for = [&](int tiles, bool pair) {
        const int lim = std::max(1, pair ? cta_cap / 2 : cta_cap);
        if (p->force_split > 0) return std::min({p->force_split, p->R, lim});
        int S = 1;
        if (tiles * 4 <= p->sm_count && p->K >= 1024) {
            S = std::min<int>(p->R, p->sm_count / tiles);
            while (S > 1 && p->K / S < 512) --S;
        }
        return std::max(1, std::min(S, lim));
    };
    const int window_mtiles = (int)std::min<int64_t>(p->Mt, (p->bn * p->cm + BM - 1) / BM);
    // The CTA-pair kernel computes 256-row tiles with one 2-CTA MMA stream; it
    // needs an even number of 128-row tiles and clusters of two resident CTAs.
    // Both halves of a pair tile are consumed in lock step, so the fused path
    // also needs every staging step of a 256-row tile resident in the ring.
    // Automatic: the fused path on pairs when the staging window holds at least
    // two pair tiles per pair of SMs, the unfused path on single CTAs.
    // Measured on GB300 (fused, with the tail split): 8192^3 442 -> 430 us on
    // pairs (its window holds 256 pair tiles); the 2048 x 4096 x 4096 and
    // 4096 x 7168 x 2048 problems (32 and 64 pair tiles in the window) 66 -> 75
    // and 82 -> 92 us; unfused 8192^3 410 -> 424 us.
    const bool pair_ok = p->allow_pair != 0 && p->Mt % 2 == 0;
    const int64_t window_pair_tiles = (int64_t)(window_mtiles / 2) * ((p->N + BN - 1) / BN);
    const bool pair_fused_fits = pair_ok && p->max_pairs_fused > 0 && p->bn >= tile_span(p->M, p->cm, 2 * BM);
    p->pair_unfused = (pair_ok && p->allow_pair == 1 && p->max_pairs_unfused > 0) ? 1 : 0;
    // (a requested 128-column tile keeps single CTAs: pair tiles are 256 wide)
    p->pair_fused = (pair_fused_fits &&
                     (p->allow_pair == 1 ||
                      (p->tile_opt != BN_NARROW &&
                       window_pair_tiles >= 2 * (int64_t)std::min(cta_cap / 2, p->max_pairs_fused))))
                        ? 1
                        : 0;
    // Tile width.  The narrow 128-column tile gives twice the work items for
    // the same rows in flight (the fused path can only work on the rows in the
    // staging ring) and double-buffers the TMEM accumulator, at 1.33x the
    // operand bytes per flop.  Measured on GB300 a K block costs nearly as much
    // time narrow as wide (the per-stage load and issue work does not shrink
    // with the tile), so the wide tile is the default and the narrow one an
    // option.  The CTA-pair kernel has wide tiles only.
    auto pick = [&](bool pair) {
        if (pair) return BN;
        return p->tile_opt ? p->tile_opt : BN;
    };
    p->tn_fused = pick(p->pair_fused);
    p->tn_unfused = pick(p->pair_unfused);
    p->Nt_fused = (int)((p->N + p->tn_fused - 1) / p->tn_fused);
    p->Nt_unfused = (int)((p->N + p->tn_unfused - 1) / p->tn_unfused);
    p->S_fused = split_for(window_mtiles * p->Nt_fused, p->pair_fused);
    p->S_unfused = split_for(p->Mt * p->Nt_unfused, p->pair_unfused);
    p->W_fused = (p->pair_fused ? p->Mt / 2 : p->Mt) * p->Nt_fused * p->S_fused;
    p->W_unfused = (p->pair_unfused ? p->Mt / 2 : p->Mt) * p->Nt_unfused * p->S_unfused;
    // Raster groups (m rows processed n-tile outer inside a group).  Unfused:
    // up to group_cap m rows, so the CTAs in flight share a few B tiles and A
    // rows in L2.  Fused: one m row.  A fused group must be whole staging
    // steps that fit in the ring, and its slots then drain together only when
    // its last items finish; measured on GB300 that stall costs more than the
    // L2 reuse gains, so the fused path consumes the steps one m-tile at a time.
    {
        const int row_u = p->pair_unfused ? 2 * BM : BM;
        const int rows_u = (int)((p->M + row_u - 1) / row_u);
        p->group_unfused = std::max(1, std::min(rows_u, p->group_cap));
        p->group_fused = 1;
        // Option: a fused group of g m-tiles, which must keep the items' order
        // monotone in staging steps at group granularity (the credit protocol's
        // freedom from deadlock rests on it): g divides the m-tiles of a step, or
        // is a multiple of them within the ring's rows.
        // Default (option 0): half the ring's steps, so that the other half can be
        // staged while a group is read (measured on the 8192^3 workload on GB300:
        // DRAM reads 1.07 GB -> 0.39 GB per launch, 2-4 % faster).
        // The CTA-pair kernel's m rows are pairs of m-tiles: the same rule in
        // units of 256 rows (commMSize a multiple of 256).
        const int row_f = p->pair_fused ? 2 * BM : BM;
        int g = p->group_fused_opt;
        if (g == 0 && p->cm % BM == 0) g = std::max(1, p->bn / 2) * (int)(p->cm / BM);
        if (p->pair_fused) g /= 2;
        if (g > 1 && p->cm % row_f == 0) {
            const int tps = (int)(p->cm / row_f);                       // m rows per step
            const int ring = (int)((int64_t)p->bn * p->cm / row_f);     // m rows in the ring
            int gg = 1;
            if (g <= tps) {
                for (int d = g; d >= 1; --d)
                    if (tps % d == 0) { gg = d; break; }
            } else {
                gg = std::min(g / tps, ring / tps) * tps;
            }
            p->group_fused = std::max(1, std::min(gg, p->pair_fused ? p->Mt / 2 : p->Mt));
        }
    }
    // Staging copy chunk: the largest divisor of commMSize rows within the
    // chunk size.  Automatic: about two steps' tasks for all copy workers (a
    // drained segment is then copied by many workers at once), 4..16 KiB
    // (smaller chunks cost more per byte, larger ones fewer copiers).
    int64_t chunk = p->chunk_bytes;
    if (chunk <= 0) {
        const int64_t step_bytes = (int64_t)p->R * p->cm * p->ka;
        chunk = std::min<int64_t>(16384, std::max<int64_t>(4096, 2 * step_bytes / ((int64_t)kCopyWarps * p->sm_count)));
    }
    int64_t want = std::max<int64_t>(1, chunk / p->ka);
    int rpc = 1;
    for (int64_t d = 1; d <= p->cm; ++d)
        if (p->cm % d == 0 && d <= want) rpc = (int)d;
    p->rows_per_chunk = rpc;
    p->chunks_per_seg = (int)(p->cm / rpc);
    p->n_copy_tasks = p->steps * p->R * p->chunks_per_seg;
    int cap = p->sm_count;
    if (p->grid_cap > 0) cap = std::min(cap, p->grid_cap);
    if (p->pair_fused) {
        const int pf = std::min(cap / 2, p->max_pairs_fused);
        p->grid_fused = 2 * std::max(1, std::min(pf, std::max(p->W_fused, (p->n_copy_tasks + 1) / 2)));
    } else {
        p->grid_fused = std::max(1, std::min(cap, std::max(p->W_fused, p->n_copy_tasks)));
    }
    if (p->pair_unfused) {
        const int pu = std::min(cap / 2, p->max_pairs_unfused);
        p->grid_unfused = 2 * std::max(1, std::min(pu, p->W_unfused));
    } else {
        p->grid_unfused = std::max(1, std::min(cap, p->W_unfused));
    }
    // Tail split (no uniform split): when the tiles fill the persistent grid
    // (its CTAs, or CTA pairs) more than once, the last round holds rem of them
    // and leaves the others idle.  If rem is at most half the grid,
    // those tiles are split in two along K (R even, each half reading R / 2
    // segments), so that the last round takes half a tile.  A split costs a
    // fixed epilogue: measured on GB300 (8192^3, traced) about 3.6 us to write
    // the fp32 partial, 1 us waiting for the other half and 2.5 us for the sum,
    // against 13.6 us of MMAs saved; so only where a half tile has at least
    // 32 K blocks (K >= 8192).  Quarter splits of 4096-deep tiles measured
    // 16-27 us slower than whole tiles.
    auto tail = [&](int& W, int S, int grid, bool pair, int& Wdp, int& St) {
        Wdp = W;
        St = 1;
        const int units = pair ? grid / 2 : grid;   // CTAs, or CTA pairs, that take items
        if (!p->tail_split || S != 1 || W <= units || p->R % 2 != 0 || p->K < 8192) return;
        const int rem = W % units;
        if (rem == 0 || 2 * rem > units) return;
        St = 2;
        Wdp = W - rem;
        W = Wdp + rem * St;
    };
    tail(p->W_fused, p->S_fused, p->grid_fused, p->pair_fused, p->Wdp_fused, p->St_fused);
    tail(p->W_unfused, p->S_unfused, p->grid_unfused, p->pair_unfused, p->Wdp_unfused, p->St_unfused);
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// The device address of pinned (page-locked) host memory, or NULL for any
// other pointer (pageable host memory is left to the DMA copies).
const void* host_device_view(const void* h) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int check_device(mxa2a_plan* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MXA2A_ERR_CUDA;
    if (dev != p->device) return MXA2A_ERR_WRONG_DEVICE;
    return MXA2A_OK;
}

int check_args(mxa2a_plan* p, const void* const* A_seg, const void* const* A_sf, const void* B, const void* B_sf,
               const void* C) {
    if (!p || !A_seg || !A_sf || !B || !B_sf || !C) return MXA2A_ERR_NULL_PTR;
    for (int r = 0; r < p->nseg; ++r) {
        if (!A_seg[r] || !A_sf[r]) return MXA2A_ERR_NULL_PTR;
        if (!aligned(A_seg[r], 16) || !aligned(A_sf[r], 4)) return MXA2A_ERR_MISALIGNED;
    }
    if (!aligned(B, 16) || !aligned(C, 16) || !aligned(B_sf, 4)) return MXA2A_ERR_MISALIGNED;
    return MXA2A_OK;
}

void fill_params(mxa2a_plan* p, GemmParams& g, const void* const* A_seg, const void* const* A_sf, void* C,
                 bool fused) {
    std::memset(&g, 0, sizeof g);
    g.R = p->R;
    g.M = (int)p->M;
    g.N = (int)p->N;
    g.ka = (int)p->ka;
    g.K = (int)p->K;
    g.cm = (int)p->cm;
    g.bn = p->bn;
    g.steps = p->steps;
    g.Mt = p->Mt;
    g.Nt = fused ? p->Nt_fused : p->Nt_unfused;
    g.tile_n = fused ? p->tn_fused : p->tn_unfused;
    // the pages' four kernel entries: E4M3E4M3, E5M2E5M2, E4M3E5M2, E5M2E4M3
    static const int kFmtA[4] = {0, 1, 0, 1}, kFmtB[4] = {0, 1, 1, 0};
    g.fmt_a = kFmtA[p->elem_types];
    g.fmt_b = kFmtB[p->elem_types];
    g.S = fused ? p->S_fused : p->S_unfused;
    g.W = fused ? p->W_fused : p->W_unfused;
    g.W_dp = fused ? p->Wdp_fused : p->Wdp_unfused;
    g.S_tail = fused ? p->St_fused : p->St_unfused;
    g.pair = fused ? p->pair_fused : p->pair_unfused;
    g.group_m = fused ? p->group_fused : p->group_unfused;
    g.kb_per_seg = (int)(p->ka / BK);
    g.Mg = p->Mg;
    g.Ng2 = p->Ng2;
    g.box_m = p->box_m;
    g.zigzag = p->zigzag;
    g.rotate = p->rotate;
    g.sfa = p->sfa;
    g.sfb = p->sfb;
    g.C = static_cast<uint16_t*>(C);
    g.partial = p->partial;
    g.ready = p->ready;
    g.fused = fused ? 1 : 0;
    g.exchange_only = fused ? p->exchange_only : 0;
    g.rows_per_chunk = p->rows_per_chunk;
    g.chunks_per_seg = p->chunks_per_seg;
    g.n_copy_tasks = p->n_copy_tasks;
    g.fault_skip_step = p->fault_skip_step;
    g.step_credits = p->step_credits;
    g.copy_skew_ns = p->copy_skew_ns;
    g.ring = p->ring;
    g.sfa_stage = p->sfa;
    g.flags = p->flags;
    g.status = p->status;
    g.launch_id = ++p->launch_id;
    g.timeout_ns = p->timeout_ns;
    g.seg_rows = (int)p->seg_rows;
    for (int r = 0; r < p->nseg; ++r) {
        g.A_seg[r] = static_cast<const uint8_t*>(A_seg[r]);
        g.A_sf_seg[r] = static_cast<const uint8_t*>(A_sf[r]);
    }
}

int refresh_b_map(mxa2a_plan* p, const void* B) {
    if (p->tmap_b_ptr == B) return MXA2A_OK;
    if (!encode_2d(&p->tmap_b, B, (uint64_t)p->K, (uint64_t)p->N, BN) ||
        !encode_2d(&p->tmap_b_half, B, (uint64_t)p->K, (uint64_t)p->N, BN / 2))
        return MXA2A_ERR_CUDA;
    p->tmap_b_ptr = B;
    return MXA2A_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MXA2A_OK : MXA2A_ERR_CUDA; }

// (Re)allocate the split-K scratch for the plan's current splits (zeroed).
int ensure_partials(mxa2a_plan* p) {
    const int S = std::max(p->S_fused, p->S_unfused);
    // partials of the tail split: one per tail item and CTA (two CTAs per item in a pair)
    const size_t tail_items = 2 * (size_t)std::max(p->W_fused - p->Wdp_fused, p->W_unfused - p->Wdp_unfused);
    if (S <= 1 && tail_items == 0) return MXA2A_OK;
    // tile t of a path's Mt x Nt tiles holds S partials of BM x tile_n floats;
    // Nt * tile_n <= Ng2 * 128 for both tile widths
    const size_t tiles = (size_t)p->Mt * std::max(p->Nt_fused, p->Nt_unfused);
    const size_t part = std::max((size_t)p->Mt * S * BM * ((size_t)p->Ng2 * 128), tail_items * BM * BN) * sizeof(float);
    const size_t rdy = std::max(tiles * S, tail_items) * sizeof(unsigned long long);
    const size_t need = part + rdy;
    if (need <= p->partial_bytes) return MXA2A_OK;
    if (p->split_ws) cudaFree(p->split_ws);
    p->split_ws = nullptr;
    p->partial = nullptr;
    p->partial_bytes = 0;
    if (cudaMalloc(reinterpret_cast<void**>(&p->split_ws), need) != cudaSuccess ||
        cudaMemset(p->split_ws + part, 0, rdy) != cudaSuccess) {
        cudaGetLastError();
        if (p->split_ws) cudaFree(p->split_ws);
        p->split_ws = nullptr;
        return MXA2A_ERR_CUDA;
    }
    p->partial = reinterpret_cast<float*>(p->split_ws);
    p->ready = reinterpret_cast<unsigned long long*>(p->split_ws + part);
    p->partial_bytes = need;
    return MXA2A_OK;
}

enum RunMode { kRunFused, kRunUnfused, kRunDirect };

// The collective side of one GEMM + ReduceScatter or GEMM + AllReduce run.
struct RsRun {
    bool fused;                 // the GEMM's epilogue routes and sums (else the reduce kernel after it)
    const void* const* recv;    // rs_R entries (entry rs_rank unused)
    void* const* send;          // rs_nblk entries (entry rs_own unused); NULL for the all-reduce
    void* pub;                  // the all-reduce's published partial, else NULL
    void* out;
};

bool is_rs_kind(const mxa2a_plan* p) {
    return p->kind == MXA2A_KIND_REDUCE_SCATTER || p->kind == MXA2A_KIND_ALLREDUCE;
}

int run_impl(mxa2a_plan* p, const void* const* A_seg, const void* const* A_sf, const void* B, const void* B_sf,
             void* C, void* stream_v, RunMode mode, const RsRun* rs = nullptr) {
    const bool fused = mode == kRunFused;
    int rc = check_args(p, A_seg, A_sf, B, B_sf, C);
    if (rc) return rc;
    // a reduce-scatter plan runs through its own calls only, and they through this path with A read in place
    if (is_rs_kind(p) != (rs != nullptr) || (rs && mode != kRunDirect))
        return MXA2A_ERR_INVALID_OPTION;
    if ((rc = check_device(p))) return rc;
    if ((rc = refresh_b_map(p, B))) return rc;
    const bool rs_fused = rs && rs->fused;
    if (rs_fused) {
        if (p->tmap_out_ptr != C) {
            if (!encode_c(&p->tmap_out, C, (uint64_t)p->rs_rows, (uint64_t)p->N)) return MXA2A_ERR_CUDA;
            p->tmap_out_ptr = C;
        }
    } else if (p->tmap_c_ptr != C) {
        if (!encode_c(&p->tmap_c, C, (uint64_t)p->M, (uint64_t)p->N)) return MXA2A_ERR_CUDA;
        p->tmap_c_ptr = C;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    int launches = 0;
    GemmParams g;
    fill_params(p, g, A_seg, A_sf, C, fused);
    g.c_host = rs ? nullptr : static_cast<uint16_t*>(p->c_host);
    if (mode == kRunDirect) {
        // the single-CTA GEMM reading A in place: one tensor map per segment,
        // re-encoded and copied to the workspace when the segment pointers change
        if (g.pair) return MXA2A_ERR_INVALID_OPTION;
        // all-gather: every 128-row tile must sit inside one input block
        if (p->seg_rows % BM) return MXA2A_ERR_INVALID_OPTION;
        const uint64_t rows = p->seg_rows ? (uint64_t)p->seg_rows : (uint64_t)p->M;
        const uint64_t cols = p->seg_rows ? (uint64_t)p->K : (uint64_t)p->ka;   // an input buffer's row
        bool same = true;
        for (int r = 0; r < p->nseg; ++r) same = same && p->seg_ptrs[r] == A_seg[r];
        if (!same) {
            for (int r = 0; r < p->nseg; ++r) {
                if (!encode_2d(&p->seg_maps_host[r], A_seg[r], cols, rows, BM))
                    return MXA2A_ERR_CUDA;
                p->seg_ptrs[r] = A_seg[r];
            }
            if ((rc = cuda_rc(cudaMemcpyAsync(p->seg_maps_dev, p->seg_maps_host, sizeof(CUtensorMap) * p->nseg,
                                              cudaMemcpyHostToDevice, stream))))
                return rc;
        }
        g.direct = 1;
        g.seg_maps = p->seg_maps_dev;
    }
    if (rs_fused) {
        // the epilogue stores the peers' blocks (and a published partial) through one
        // tensor map per buffer
        auto target = [&](int j) -> void* {
            if (j == p->rs_own) return p->rs_publish ? rs->pub : nullptr;
            return rs->send[j];
        };
        bool same = true;
        for (int j = 0; j < p->rs_nblk; ++j) same = same && p->send_ptrs[j] == target(j);
        if (!same) {
            for (int j = 0; j < p->rs_nblk; ++j) {
                void* t = target(j);
                if (!t) {
                    std::memset(&p->send_maps_host[j], 0, sizeof(CUtensorMap));
                } else if (!encode_c(&p->send_maps_host[j], t, (uint64_t)p->rs_rows, (uint64_t)p->N)) {
                    return MXA2A_ERR_CUDA;
                }
                p->send_ptrs[j] = t;
            }
            if ((rc = cuda_rc(cudaMemcpyAsync(p->send_maps_dev, p->send_maps_host,
                                              sizeof(CUtensorMap) * p->rs_nblk, cudaMemcpyHostToDevice, stream))))
                return rc;
        }
        g.rs_rows = (int)p->rs_rows;
        g.rs_rank = p->rs_rank;
        g.rs_R = p->rs_R;
        g.rs_own = p->rs_own;
        g.rs_publish = p->rs_publish;
        g.rs_pub = static_cast<const uint16_t*>(rs->pub);
        g.send_maps = p->send_maps_dev;
        g.rs_cnt = p->rs_cnt;
        for (int j = 0; j < p->rs_R; ++j)
            g.recv[j] = j == p->rs_rank ? nullptr : static_cast<const uint16_t*>(rs->recv[j]);
    }
    // Split partials are tagged with this run's launch index, which a graph
    // replays unchanged: a split plan must not be captured, and a captured
    // run leaves its tail whole.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MXA2A_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone && g.S > 1) return MXA2A_ERR_CAPTURE_SPLIT;
    if (cap != cudaStreamCaptureStatusNone && g.S_tail > 1) {
        g.W = g.W_dp + (g.W - g.W_dp) / g.S_tail;
        g.W_dp = g.W;
        g.S_tail = 1;
    }
    // The B scale pack runs in the GEMM kernel's prologue, whose producers then
    // wait for every CTA's slice: a cooperative launch guarantees that they are
    // all resident.  The fused CTA-pair kernel (a cluster launch) already relies
    // on that for its staging credits (its grid never exceeds the pairs that fit
    // at once) and packs inline too; the unfused one keeps the separate kernel.
    g.B_scale = static_cast<const uint8_t*>(B_sf);
    g.sfb_inline = (!g.pair || fused) ? 1 : 0;
    if (!g.sfb_inline) {
        if ((rc = cuda_rc(launch_pack_sfb(static_cast<const uint8_t*>(B_sf), (int)p->N, (int)p->K, p->Ng2, p->sfb,
                                          stream))))
            return rc;
        ++launches;
    }
    if (mode == kRunUnfused) {
        if ((rc = cuda_rc(launch_pack_a(g, p->a_packed, 0, stream)))) return rc;
        ++launches;
    }
    const int ev_slot = p->record_events ? (int)(p->ev_recorded % p->record_events) : 0;
    if (p->record_events && (rc = cuda_rc(cudaEventRecord(p->ev0[ev_slot], stream)))) return rc;
    rc = cuda_rc(launch_mxgemm(g, fused ? p->tmap_ring : p->tmap_apacked,
                               (g.pair || g.tile_n == BN_NARROW) ? p->tmap_b_half : p->tmap_b,
                               rs_fused ? p->tmap_out : p->tmap_c, fused ? p->grid_fused : p->grid_unfused, fused,
                               stream, p->tmap_sf));
    if (rc) return rc;
    ++launches;
    if (p->record_events) {
        if ((rc = cuda_rc(cudaEventRecord(p->ev1[ev_slot], stream)))) return rc;
        ++p->ev_recorded;
    }
    if (rs && !rs->fused) {
        // the collective step after the GEMM: P (in C) -> the send buffers and out
        RsArgs ra;
        std::memset(&ra, 0, sizeof ra);
        ra.P = static_cast<const uint16_t*>(C);
        for (int j = 0; j < p->rs_R; ++j)
            if (j != p->rs_rank) ra.recv[j] = static_cast<const uint16_t*>(rs->recv[j]);
        for (int j = 0; j < p->rs_nblk; ++j)
            if (j != p->rs_own) ra.send[j] = static_cast<uint16_t*>(rs->send[j]);
        ra.out = static_cast<uint16_t*>(rs->out);
        ra.R = p->rs_R;
        ra.rank = p->rs_rank;
        ra.rows = (int)p->rs_rows;
        ra.N = (int)p->N;
        ra.nblk = p->rs_nblk;
        ra.own = p->rs_own;
        if ((rc = cuda_rc(launch_rs_reduce(ra, stream)))) return rc;
        ++launches;
    }
    p->last_launches = launches;
    return MXA2A_OK;
}

mxa2a_plan* create_impl(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num,
                        int kind, int nseg, int64_t seg_rows, bool staging = true) {
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        g_last_error = MXA2A_ERR_CUDA;
        return nullptr;
    }
    if (major != 10 || minor != 3) {
        g_last_error = MXA2A_ERR_UNSUPPORTED_DEVICE;
        return nullptr;
    }
    mxa2a_plan* p = new (std::nothrow) mxa2a_plan();
    if (!p) {
        g_last_error = MXA2A_ERR_CUDA;
        return nullptr;
    }
    p->R = R;
    p->kind = kind;
    p->nseg = nseg;
    p->seg_rows = seg_rows;
    p->M = M;
    p->ka = kPerRank;
    p->N = N;
    p->cm = commMSize;
    p->bn = buffer_num;
    p->device = dev;
    p->sm_count = sms;
    p->max_pairs_fused = mxgemm_max_pairs(true);
    p->max_pairs_unfused = mxgemm_max_pairs(false);
    derive(p);
    // workspace: ring | sfa | sfb | packed A | flags | status (split-K partials separately)
    // (a plan that reads A in place only has no ring and no packed A)
    p->ring_bytes = staging ? (size_t)buffer_num * R * commMSize * kPerRank : 0;
    p->sfa_bytes = (size_t)(p->K / BK) * p->Mg * kSfAtomBytes;
    p->sfb_bytes = (size_t)(p->K / BK) * p->Ng2 * kSfAtomBytes;
    p->apacked_bytes = staging ? (size_t)M * p->K : 0;
    p->flags_bytes = FlagLayout::words(buffer_num, R) * sizeof(unsigned long long);
    size_t off = 0;
    const size_t o_ring = off; off = align_up(off + p->ring_bytes, 1024);
    const size_t o_sfa = off; off = align_up(off + p->sfa_bytes, 1024);
    const size_t o_sfb = off; off = align_up(off + p->sfb_bytes, 1024);
    const size_t o_ap = off; off = align_up(off + p->apacked_bytes, 1024);
    const size_t o_flags = off; off = align_up(off + p->flags_bytes, 1024);
    const size_t o_status = off; off = align_up(off + sizeof(DevStatus), 1024);
    const size_t o_maps = off; off = align_up(off + sizeof(CUtensorMap) * 2 * kMaxSegments, 1024);
    // reduce-scatter tile counts, for either tile width (the narrow tile has 2 Nt columns of tiles)
    p->rs_cnt_bytes = (kind == MXA2A_KIND_REDUCE_SCATTER || kind == MXA2A_KIND_ALLREDUCE)
                          ? (size_t)p->Mt * 2 * p->Nt * sizeof(unsigned long long)
                          : 0;
    const size_t o_rs = off; off = align_up(off + p->rs_cnt_bytes, 1024);
    p->ws_bytes = off;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        g_last_error = MXA2A_ERR_CUDA;
        return nullptr;
    }
    p->ring = p->ws + o_ring;
    p->sfa = p->ws + o_sfa;
    p->sfb = p->ws + o_sfb;
    p->a_packed = p->ws + o_ap;
    p->flags = reinterpret_cast<unsigned long long*>(p->ws + o_flags);
    p->status = reinterpret_cast<DevStatus*>(p->ws + o_status);
    p->seg_maps_dev = reinterpret_cast<CUtensorMap*>(p->ws + o_maps);
    p->send_maps_dev = p->seg_maps_dev + kMaxSegments;
    p->rs_cnt = p->rs_cnt_bytes ? reinterpret_cast<unsigned long long*>(p->ws + o_rs) : nullptr;
    bool ok = cudaMemset(p->ws + o_sfa, 0, p->sfa_bytes) == cudaSuccess &&
              cudaMemset(p->flags, 0, p->flags_bytes) == cudaSuccess &&
              cudaMemset(p->status, 0, sizeof(DevStatus)) == cudaSuccess &&
              (!p->rs_cnt_bytes || cudaMemset(p->rs_cnt, 0, p->rs_cnt_bytes) == cudaSuccess) &&
              ensure_partials(p) == MXA2A_OK;
    if (staging) {
        ok = ok && encode_2d(&p->tmap_ring, p->ring, (uint64_t)kPerRank, (uint64_t)buffer_num * R * commMSize,
                             (uint32_t)p->box_m);
        ok = ok && encode_2d(&p->tmap_apacked, p->a_packed, (uint64_t)p->K, (uint64_t)M, BM);
    } else {
        std::memset(&p->tmap_ring, 0, sizeof(CUtensorMap));      // never used: A is read in place
        std::memset(&p->tmap_apacked, 0, sizeof(CUtensorMap));
    }
    ok = ok && encode_atoms(&p->tmap_sf[0], p->sfa, (uint64_t)(p->K / BK) * p->Mg, 2) &&
         encode_atoms(&p->tmap_sf[1], p->sfb, (uint64_t)(p->K / BK) * p->Ng2, 4);
    if (!ok || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        mxa2a_destroy(p);
        g_last_error = MXA2A_ERR_CUDA;
        return nullptr;
    }
    g_last_error = MXA2A_OK;
    return p;
}

}  // namespace

extern "C" {

int mxa2a_validate(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num) {
    if (R < 1 || R > kMaxSegments) return MXA2A_ERR_INVALID_SHAPE;
    if (M < 1 || kPerRank < BK || N < 16 || commMSize < 64) return MXA2A_ERR_INVALID_SHAPE;
    if (kPerRank % BK || N % 16 || commMSize % 64 || M % commMSize) return MXA2A_ERR_INVALID_SHAPE;
    if (buffer_num < 1 || buffer_num > 8) return MXA2A_ERR_INVALID_SHAPE;
    const int64_t lim = int64_t(1) << 20;
    if (M > lim || N > lim || (int64_t)R * kPerRank > lim) return MXA2A_ERR_INVALID_SHAPE;
    if (buffer_num < tile_span(M, commMSize)) return MXA2A_ERR_INVALID_SHAPE;
    return MXA2A_OK;
}

int mxa2a_last_error(void) { return g_last_error; }

mxa2a_plan* mxa2a_create(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num) {
    const int rc = mxa2a_validate(R, M, kPerRank, N, commMSize, buffer_num);
    if (rc) {
        g_last_error = rc;
        return nullptr;
    }
    return create_impl(R, M, kPerRank, N, commMSize, buffer_num, MXA2A_KIND_ALLTOALL, R, 0);
}

int mxa2a_validate_allgather(int R, int64_t rowsPerRank, int64_t K, int64_t N, int64_t commMSize, int buffer_num) {
    if (R < 1 || R > kMaxSegments || rowsPerRank < 1 || commMSize < 1) return MXA2A_ERR_INVALID_SHAPE;
    if (rowsPerRank % commMSize || (int64_t)R * rowsPerRank > (int64_t(1) << 20)) return MXA2A_ERR_INVALID_SHAPE;
    return mxa2a_validate(1, (int64_t)R * rowsPerRank, K, N, commMSize, buffer_num);
}

int mxa2a_validate_reduce_scatter(int R, int rank, int64_t M, int64_t K, int64_t N) {
    if (R < 1 || R > kMaxSegments || rank < 0 || rank >= R) return MXA2A_ERR_INVALID_SHAPE;
    if (M < 64 * (int64_t)R || M % (64 * (int64_t)R)) return MXA2A_ERR_INVALID_SHAPE;
    return mxa2a_validate(1, M, K, N, 64, 2);
}

mxa2a_plan* mxa2a_create_reduce_scatter(int R, int rank, int64_t M, int64_t K, int64_t N) {
    const int rc = mxa2a_validate_reduce_scatter(R, rank, M, K, N);
    if (rc) {
        g_last_error = rc;
        return nullptr;
    }
    // one K slice, A read in place (no staging ring, no packed A)
    mxa2a_plan* p = create_impl(1, M, K, N, 64, 2, MXA2A_KIND_REDUCE_SCATTER, 1, 0, false);
    if (p) {
        p->rs_rank = rank;
        p->rs_R = R;
        p->rs_rows = M / R;
        p->rs_nblk = R;
        p->rs_own = rank;
        p->rs_publish = 0;
    }
    return p;
}

int mxa2a_validate_allreduce(int R, int rank, int64_t M, int64_t K, int64_t N) {
    if (R < 1 || R > kMaxSegments || rank < 0 || rank >= R) return MXA2A_ERR_INVALID_SHAPE;
    return mxa2a_validate(1, M, K, N, 64, 2);
}

mxa2a_plan* mxa2a_create_allreduce(int R, int rank, int64_t M, int64_t K, int64_t N) {
    const int rc = mxa2a_validate_allreduce(R, rank, M, K, N);
    if (rc) {
        g_last_error = rc;
        return nullptr;
    }
    mxa2a_plan* p = create_impl(1, M, K, N, 64, 2, MXA2A_KIND_ALLREDUCE, 1, 0, false);
    if (p) {   // one block of all M rows, summed here and published
        p->rs_rank = rank;
        p->rs_R = R;
        p->rs_rows = M;
        p->rs_nblk = 1;
        p->rs_own = 0;
        p->rs_publish = 1;
    }
    return p;
}

namespace {
int run_rs(mxa2a_plan* p, const void* A, const void* A_sf, const void* B, const void* B_sf, const void* const* recv,
           void* const* send, void* out, void* stream, bool fused) {
    if (!p || !recv || !send || !out) return MXA2A_ERR_NULL_PTR;
    if (p->kind != MXA2A_KIND_REDUCE_SCATTER) return MXA2A_ERR_INVALID_OPTION;
    for (int j = 0; j < p->rs_R; ++j) {
        if (j == p->rs_rank) continue;
        if (!recv[j] || !send[j]) return MXA2A_ERR_NULL_PTR;
        if (!aligned(recv[j], 16) || !aligned(send[j], 16)) return MXA2A_ERR_MISALIGNED;
    }
    if (!aligned(out, 16)) return MXA2A_ERR_MISALIGNED;
    void* C = out;
    if (!fused) {
        int rc = check_device(p);
        if (rc) return rc;
        if (!p->rs_scratch) {
            if (cudaMalloc(&p->rs_scratch, (size_t)p->M * p->N * 2) != cudaSuccess) {
                cudaGetLastError();
                p->rs_scratch = nullptr;
                return MXA2A_ERR_CUDA;
            }
        }
        C = p->rs_scratch;
    }
    const RsRun rs{fused, recv, send, nullptr, out};
    const void* a_seg[1] = {A};
    const void* a_sf[1] = {A_sf};
    return run_impl(p, a_seg, a_sf, B, B_sf, C, stream, kRunDirect, &rs);
}

int run_ar(mxa2a_plan* p, const void* A, const void* A_sf, const void* B, const void* B_sf, const void* const* recv,
           void* pub, void* out, void* stream, bool fused) {
    if (!p || !recv || !pub || !out) return MXA2A_ERR_NULL_PTR;
    if (p->kind != MXA2A_KIND_ALLREDUCE) return MXA2A_ERR_INVALID_OPTION;
    for (int j = 0; j < p->rs_R; ++j) {
        if (j == p->rs_rank) continue;
        if (!recv[j]) return MXA2A_ERR_NULL_PTR;
        if (!aligned(recv[j], 16)) return MXA2A_ERR_MISALIGNED;
    }
    if (!aligned(out, 16) || !aligned(pub, 16)) return MXA2A_ERR_MISALIGNED;
    // fused: the GEMM's epilogue publishes the partial and the kernel sums into
    // out; unfused: the GEMM writes the partial into pub, then the reduce kernel
    const RsRun rs{fused, recv, nullptr, pub, out};
    const void* a_seg[1] = {A};
    const void* a_sf[1] = {A_sf};
    return run_impl(p, a_seg, a_sf, B, B_sf, fused ? out : pub, stream, kRunDirect, &rs);
}
}  // namespace

int mxa2a_run_allreduce(mxa2a_plan* p, const void* A, const void* A_sf, const void* B, const void* B_sf,
                        const void* const* recv, void* pub, void* out, void* stream) {
    return run_ar(p, A, A_sf, B, B_sf, recv, pub, out, stream, true);
}

int mxa2a_run_allreduce_unfused(mxa2a_plan* p, const void* A, const void* A_sf, const void* B, const void* B_sf,
                                const void* const* recv, void* pub, void* out, void* stream) {
    return run_ar(p, A, A_sf, B, B_sf, recv, pub, out, stream, false);
}

int mxa2a_run_reduce_scatter(mxa2a_plan* p, const void* A, const void* A_sf, const void* B, const void* B_sf,
                             const void* const* recv, void* const* send, void* out, void* stream) {
    return run_rs(p, A, A_sf, B, B_sf, recv, send, out, stream, true);
}

int mxa2a_run_reduce_scatter_unfused(mxa2a_plan* p, const void* A, const void* A_sf, const void* B,
                                     const void* B_sf, const void* const* recv, void* const* send, void* out,
                                     void* stream) {
    return run_rs(p, A, A_sf, B, B_sf, recv, send, out, stream, false);
}

mxa2a_plan* mxa2a_create_allgather(int R, int64_t rowsPerRank, int64_t K, int64_t N, int64_t commMSize,
                                   int buffer_num) {
    const int rc = mxa2a_validate_allgather(R, rowsPerRank, K, N, commMSize, buffer_num);
    if (rc) {
        g_last_error = rc;
        return nullptr;
    }
    // The staging ring carries K slices of the gathered rows, as it carries the
    // all-to-all's segments: credits per (slot, slice) let a slice of the next
    // step land while other slices of the slot are still being read.  Slices
    // of about 1024 columns (at least 8 K blocks each), at most 64.
    const int64_t kb = K / BK;
    int slices = 1;
    for (int64_t d = 1; d <= std::min<int64_t>(kMaxSegments, kb / 8); ++d)
        if (kb % d == 0) slices = (int)d;
    // the copy role and the pack pick the input block by row and the columns by slice
    return create_impl(slices, (int64_t)R * rowsPerRank, K / slices, N, commMSize, buffer_num,
                       MXA2A_KIND_ALLGATHER, R, rowsPerRank);
}

int mxa2a_run(mxa2a_plan* p, const void* const* A_seg, const void* const* A_sf, const void* B, const void* B_sf,
              void* C, void* stream) {
    return run_impl(p, A_seg, A_sf, B, B_sf, C, stream, kRunFused);
}

int mxa2a_run_unfused(mxa2a_plan* p, const void* const* A_seg, const void* const* A_sf, const void* B,
                      const void* B_sf, void* C, void* stream) {
    return run_impl(p, A_seg, A_sf, B, B_sf, C, stream, kRunUnfused);
}

int mxa2a_run_direct(mxa2a_plan* p, const void* const* A_seg, const void* const* A_sf, const void* B,
                     const void* B_sf, void* C, void* stream) {
    return run_impl(p, A_seg, A_sf, B, B_sf, C, stream, kRunDirect);
}

int mxa2a_run_host(mxa2a_plan* p, const void* const* A_seg_h, const void* const* A_sf_h, const void* B_h,
                   const void* B_sf_h, void* C_h, void* stream_v) {
    if (!p || !A_seg_h || !A_sf_h || !B_h || !B_sf_h || !C_h) return MXA2A_ERR_NULL_PTR;
    for (int r = 0; r < p->nseg; ++r)
        if (!A_seg_h[r] || !A_sf_h[r]) return MXA2A_ERR_NULL_PTR;
    int rc = check_device(p);
    if (rc) return rc;
    const size_t seg_m = p->seg_rows ? (size_t)p->seg_rows : (size_t)p->M;
    const size_t seg_k = p->seg_rows ? (size_t)p->K : (size_t)p->ka;
    const size_t a_b = seg_m * seg_k, asf_b = seg_m * (seg_k / 32);
    const size_t b_b = (size_t)p->N * p->K, bsf_b = (size_t)p->N * (p->K / 32), c_b = (size_t)p->M * p->N * 2;
    const size_t a_s = align_up(a_b, 256), asf_s = align_up(asf_b, 256);
    const size_t need = p->nseg * (a_s + asf_s) + align_up(b_b, 256) + align_up(bsf_b, 256) + align_up(c_b, 256);
    if (p->io_bytes < need) {
        if (p->io) cudaFree(p->io);
        p->io = nullptr;
        p->io_bytes = 0;
        if (cudaMalloc(&p->io, need) != cudaSuccess) {
            cudaGetLastError();
            return MXA2A_ERR_CUDA;
        }
        p->io_bytes = need;
        p->tmap_b_ptr = nullptr;
        p->tmap_c_ptr = nullptr;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream_v);
    const void* dA[kMaxSegments];
    const void* dS[kMaxSegments];
    const void* src[2 * kMaxSegments + 2];
    void* dst[2 * kMaxSegments + 2];
    size_t len[2 * kMaxSegments + 2];
    int n = 0;
    uint8_t* cur = p->io;
    // Pinned segments are read in place by the fused kernel's staging copies
    // (the exchange then reads host memory through the device's link to it).
    bool a_in_place = true;
    for (int r = 0; r < p->nseg && a_in_place; ++r) {
        dA[r] = host_device_view(A_seg_h[r]);
        dS[r] = host_device_view(A_sf_h[r]);
        a_in_place = dA[r] && dS[r] && aligned(dA[r], 16) && aligned(dS[r], 4);
    }
    for (int r = 0; r < p->nseg; ++r) {
        if (!a_in_place) {
            dA[r] = cur;
            src[n] = A_seg_h[r], dst[n] = cur, len[n++] = a_b;
        }
        cur += a_s;
        if (!a_in_place) {
            dS[r] = cur;
            src[n] = A_sf_h[r], dst[n] = cur, len[n++] = asf_b;
        }
        cur += asf_s;
    }
    uint8_t* dB = cur;
    cur += align_up(b_b, 256);
    uint8_t* dBs = cur;
    cur += align_up(bsf_b, 256);
    uint8_t* dC = cur;
    src[n] = B_h, dst[n] = dB, len[n++] = b_b;
    src[n] = B_sf_h, dst[n] = dBs, len[n++] = bsf_b;
    // Pinned host buffers are copied by the SMs in one launch (the device reads
    // them through their device addresses); otherwise one DMA copy per buffer.
    const void* view[2 * kMaxSegments + 2];
    bool by_sms = true;
    for (int i = 0; i < n && by_sms; ++i) {
        view[i] = host_device_view(src[i]);
        by_sms = view[i] && aligned(view[i], 16) && len[i] % 16 == 0;
    }
    if (by_sms) {
        if ((rc = cuda_rc(launch_copy_list(n, view, dst, len, s)))) return rc;
    } else {
        for (int i = 0; i < n; ++i)
            if (cudaMemcpyAsync(dst[i], src[i], len[i], cudaMemcpyHostToDevice, s) != cudaSuccess)
                return MXA2A_ERR_CUDA;
    }
    // A pinned C is written by the epilogue itself, tile by tile, through its
    // device view: the host link carries C while the GEMM runs.  Otherwise
    // one DMA copy after the run.
    void* c_view = const_cast<void*>(host_device_view(C_h));
    const bool c_direct = c_view && aligned(c_view, 16);
    // With C written over the host link the automatic choice takes single CTAs:
    // measured on GB300 (8192^3, pinned buffers) 1197 us per step end to end
    // against 1222 us on CTA pairs.  The plan is derived again for this run.
    const bool single = c_direct && p->allow_pair == 2 && p->pair_fused;
    if (single) {
        p->allow_pair = 0;
        derive(p);
        rc = ensure_partials(p);
    }
    p->c_host = c_direct ? c_view : nullptr;
    if (!rc) rc = run_impl(p, dA, dS, dB, dBs, dC, stream_v, kRunFused);
    p->c_host = nullptr;
    if (single) {
        p->allow_pair = 2;
        derive(p);
    }
    if (rc) return rc;
    if (!c_direct && cudaMemcpyAsync(C_h, dC, c_b, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MXA2A_ERR_CUDA;
    return MXA2A_OK;
}

int mxa2a_get_status(mxa2a_plan* p, mxa2a_status* out) {
    if (!p || !out) return MXA2A_ERR_NULL_PTR;
    int rc = check_device(p);
    if (rc) return rc;
    DevStatus st;
    if (cudaMemcpy(&st, p->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return MXA2A_ERR_CUDA;
    std::memset(out, 0, sizeof *out);
    const unsigned long long launch = st.key >> 8;
    const int code = (int)(st.key & 0xFF);
    if (code != 0 && launch > p->checked_launch) {
        out->code = code;
        out->role = st.role;
        out->block = st.block;
        out->step = st.step;
        out->segment = st.segment;
        out->slot = st.slot;
        out->observed = st.observed;
        out->expected = st.expected;
        out->launch = (int64_t)launch;
    } else {
        out->step = out->segment = out->slot = -1;
    }
    p->checked_launch = p->launch_id;
    return MXA2A_OK;
}

namespace {
// The options that change the plan's derived choices (validated, stored; the
// caller derives the plan again).  Not one of them: MXA2A_ERR_INVALID_OPTION.
int set_planner_option(mxa2a_plan* p, int key, int64_t v) {
    switch (key) {
        case MXA2A_OPT_SPLIT_K:
            if (v < 0 || v > p->R) return MXA2A_ERR_INVALID_OPTION;
            p->force_split = (int)v;
            break;
        case MXA2A_OPT_GRID:
            if (v < 0) return MXA2A_ERR_INVALID_OPTION;
            p->grid_cap = (int)v;
            break;
        case MXA2A_OPT_CHUNK_BYTES:
            if (v != 0 && v < 16) return MXA2A_ERR_INVALID_OPTION;
            p->chunk_bytes = v;
            break;
        case MXA2A_OPT_CTA_PAIR:
            if (v < 0 || v > 2) return MXA2A_ERR_INVALID_OPTION;
            p->allow_pair = (int)v;
            break;
        case MXA2A_OPT_GROUP_M:
            if (v < 1 || v > 4096) return MXA2A_ERR_INVALID_OPTION;
            p->group_cap = (int)v;
            break;
        case MXA2A_OPT_TILE_N:
            if (v != 0 && v != BN_NARROW && v != BN) return MXA2A_ERR_INVALID_OPTION;
            p->tile_opt = (int)v;
            break;
        case MXA2A_OPT_ELEM_TYPES:
            if (v < 0 || v > 3) return MXA2A_ERR_INVALID_OPTION;
            p->elem_types = (int)v;
            break;
        case MXA2A_OPT_STEP_CREDITS:
            if (v != 0 && v != 1) return MXA2A_ERR_INVALID_OPTION;
            p->step_credits = (int)v;
            break;
        case MXA2A_OPT_COPY_SKEW_NS:
            if (v < 0 || v > 1000000) return MXA2A_ERR_INVALID_OPTION;
            p->copy_skew_ns = (int)v;
            break;
        case MXA2A_OPT_GROUP_FUSED:
            if (v < 0 || v > 1024) return MXA2A_ERR_INVALID_OPTION;
            p->group_fused_opt = (int)v;
            break;
        case MXA2A_OPT_TAIL_SPLIT:
            if (v != 0 && v != 1) return MXA2A_ERR_INVALID_OPTION;
            p->tail_split = (int)v;
            break;
        default:
            return MXA2A_ERR_INVALID_OPTION;
    }
    return MXA2A_OK;
}

// A plan fact or option value (the body of mxa2a_get_option).
int plan_get(const mxa2a_plan* p, int key, int64_t* v) {
    switch (key) {
        case MXA2A_OPT_TIMEOUT_NS: *v = p->timeout_ns; break;
        case MXA2A_OPT_SPLIT_K: *v = p->force_split; break;
        case MXA2A_OPT_ZIGZAG: *v = p->zigzag; break;
        case MXA2A_OPT_ROTATE: *v = p->rotate; break;
        case MXA2A_OPT_RECORD_EVENTS: *v = p->record_events; break;
        case MXA2A_OPT_EXCHANGE_ONLY: *v = p->exchange_only; break;
        case MXA2A_OPT_FAULT_SKIP_STEP: *v = p->fault_skip_step; break;
        case MXA2A_OPT_GRID: *v = p->grid_cap; break;
        case MXA2A_OPT_CHUNK_BYTES: *v = p->chunk_bytes; break;
        case MXA2A_OPT_CTA_PAIR: *v = p->allow_pair; break;
        case MXA2A_OPT_GROUP_M: *v = p->group_cap; break;
        case MXA2A_OPT_TILE_N: *v = p->tile_opt; break;
        case MXA2A_OPT_ELEM_TYPES: *v = p->elem_types; break;
        case MXA2A_OPT_STEP_CREDITS: *v = p->step_credits; break;
        case MXA2A_OPT_COPY_SKEW_NS: *v = p->copy_skew_ns; break;
        case MXA2A_OPT_GROUP_FUSED: *v = p->group_fused_opt; break;
        case MXA2A_OPT_TAIL_SPLIT: *v = p->tail_split; break;
        case MXA2A_INFO_GROUP_FUSED: *v = p->group_fused; break;
        case MXA2A_INFO_GROUP_UNFUSED: *v = p->group_unfused; break;
        case MXA2A_INFO_CTA_PAIR: *v = p->pair_fused; break;
        case MXA2A_INFO_CTA_PAIR_UNFUSED: *v = p->pair_unfused; break;
        case MXA2A_INFO_STEPS: *v = p->steps; break;
        case MXA2A_INFO_MTILES: *v = p->Mt; break;
        case MXA2A_INFO_NTILES: *v = p->Nt_fused; break;
        case MXA2A_INFO_TILE_N_FUSED: *v = p->tn_fused; break;
        case MXA2A_INFO_TILE_N_UNFUSED: *v = p->tn_unfused; break;
        case MXA2A_INFO_KIND: *v = p->kind; break;
        case MXA2A_INFO_TAIL_SPLIT: *v = p->St_fused; break;
        case MXA2A_INFO_TAIL_SPLIT_UNFUSED: *v = p->St_unfused; break;
        case MXA2A_INFO_SPLITS: *v = p->S_fused; break;
        case MXA2A_INFO_ITEMS: *v = p->W_fused; break;
        case MXA2A_INFO_SPLITS_UNFUSED: *v = p->S_unfused; break;
        case MXA2A_INFO_GRID_FUSED: *v = p->grid_fused; break;
        case MXA2A_INFO_GRID_UNFUSED: *v = p->grid_unfused; break;
        case MXA2A_INFO_COPY_TASKS: *v = p->n_copy_tasks; break;
        case MXA2A_INFO_ROWS_PER_CHUNK: *v = p->rows_per_chunk; break;
        case MXA2A_INFO_WORKSPACE_BYTES: *v = (int64_t)p->ws_bytes; break;
        case MXA2A_INFO_SM_COUNT: *v = p->sm_count; break;
        case MXA2A_INFO_LAUNCHES: *v = p->last_launches; break;
        default: return MXA2A_ERR_INVALID_OPTION;
    }
    return MXA2A_OK;
}
}  // namespace

int mxa2a_set_option(mxa2a_plan* p, int key, int64_t v) {
    if (!p) return MXA2A_ERR_NULL_PTR;
    switch (key) {
        case MXA2A_OPT_TIMEOUT_NS:
            if (v < 1000) return MXA2A_ERR_INVALID_OPTION;
            p->timeout_ns = v;
            return MXA2A_OK;
        case MXA2A_OPT_ZIGZAG:
            if (v != 0 && v != 1) return MXA2A_ERR_INVALID_OPTION;
            p->zigzag = (int)v;
            return MXA2A_OK;
        case MXA2A_OPT_ROTATE:
            if (v != 0 && v != 1) return MXA2A_ERR_INVALID_OPTION;
            p->rotate = (int)v;
            return MXA2A_OK;
        case MXA2A_OPT_RECORD_EVENTS:
            if (v < 0 || v > mxa2a_plan::kEvRing) return MXA2A_ERR_INVALID_OPTION;
            if (v > p->ev_count) {
                if (!p->ev0) {
                    p->ev0 = new (std::nothrow) cudaEvent_t[mxa2a_plan::kEvRing]();
                    p->ev1 = new (std::nothrow) cudaEvent_t[mxa2a_plan::kEvRing]();
                    if (!p->ev0 || !p->ev1) return MXA2A_ERR_CUDA;
                }
                for (int i = p->ev_count; i < v; ++i) {
                    if (cudaEventCreate(&p->ev0[i]) != cudaSuccess) return MXA2A_ERR_CUDA;
                    if (cudaEventCreate(&p->ev1[i]) != cudaSuccess) {
                        cudaEventDestroy(p->ev0[i]);
                        return MXA2A_ERR_CUDA;
                    }
                    p->ev_count = i + 1;
                }
            }
            p->record_events = (int)v;
            p->ev_recorded = 0;
            return MXA2A_OK;
        case MXA2A_OPT_EXCHANGE_ONLY:
            if (v != 0 && v != 1) return MXA2A_ERR_INVALID_OPTION;
            if (v == 1 && p->bn < p->steps) return MXA2A_ERR_INVALID_OPTION;
            p->exchange_only = (int)v;
            return MXA2A_OK;
        case MXA2A_OPT_FAULT_SKIP_STEP:
            if (v < -1 || v >= p->steps) return MXA2A_ERR_INVALID_OPTION;
            p->fault_skip_step = (int)v;
            return MXA2A_OK;
        default: {
            const int rc = set_planner_option(p, key, v);
            if (rc) return rc;
        }
    }
    derive(p);
    return ensure_partials(p);
}

int mxa2a_get_option(mxa2a_plan* p, int key, int64_t* v) {
    if (!p || !v) return MXA2A_ERR_NULL_PTR;
    return plan_get(p, key, v);
}

int mxa2a_plan_preview(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize, int buffer_num,
                       int sm_count, int max_pairs_fused, int max_pairs_unfused, const int* opt_keys,
                       const int64_t* opt_values, int n_opts, const int* info_keys, int64_t* info_values,
                       int n_info) {
    const int shape = mxa2a_validate(R, M, kPerRank, N, commMSize, buffer_num);
    if (shape) return shape;
    if (sm_count < 1 || max_pairs_fused < 0 || max_pairs_unfused < 0 || n_opts < 0 || n_info < 0)
        return MXA2A_ERR_INVALID_OPTION;
    if ((n_opts > 0 && (!opt_keys || !opt_values)) || (n_info > 0 && (!info_keys || !info_values)))
        return MXA2A_ERR_NULL_PTR;
    mxa2a_plan p;   // fields only: the same derivation as a created plan's
    p.R = R;
    p.kind = MXA2A_KIND_ALLTOALL;
    p.nseg = R;
    p.M = M;
    p.ka = kPerRank;
    p.N = N;
    p.cm = commMSize;
    p.bn = buffer_num;
    p.device = -1;
    p.sm_count = sm_count;
    p.max_pairs_fused = max_pairs_fused;
    p.max_pairs_unfused = max_pairs_unfused;
    derive(&p);
    for (int i = 0; i < n_opts; ++i) {
        const int rc = set_planner_option(&p, opt_keys[i], opt_values[i]);
        if (rc) return rc;
        derive(&p);
    }
    for (int i = 0; i < n_info; ++i) {
        if (info_keys[i] == MXA2A_INFO_WORKSPACE_BYTES || info_keys[i] == MXA2A_INFO_LAUNCHES)
            return MXA2A_ERR_INVALID_OPTION;
        const int rc = plan_get(&p, info_keys[i], &info_values[i]);
        if (rc) return rc;
    }
    return MXA2A_OK;
}

int mxa2a_last_kernel_ms(mxa2a_plan* p, float* ms) {
    int n = 0;
    return mxa2a_kernel_times(p, ms, 1, &n);
}

int mxa2a_kernel_times(mxa2a_plan* p, float* ms, int max_count, int* count) {
    if (!p || !ms || !count) return MXA2A_ERR_NULL_PTR;
    *count = 0;
    if (!p->record_events || p->ev_recorded == 0 || max_count < 1) return MXA2A_ERR_INVALID_OPTION;
    const long long avail = std::min<long long>(p->ev_recorded, p->record_events);
    const int n = (int)std::min<long long>(avail, max_count);
    for (int i = 0; i < n; ++i) {
        // oldest first among the last n runs
        const long long run = p->ev_recorded - n + i;
        const int slot = (int)(run % p->record_events);
        if (cudaEventSynchronize(p->ev1[slot]) != cudaSuccess) return MXA2A_ERR_CUDA;
        if (cudaEventElapsedTime(&ms[i], p->ev0[slot], p->ev1[slot]) != cudaSuccess) return MXA2A_ERR_CUDA;
    }
    *count = n;
    return MXA2A_OK;
}

int mxa2a_read_workspace(mxa2a_plan* p, int which, void* dst, size_t bytes, size_t* bytes_out) {
    if (!p) return MXA2A_ERR_NULL_PTR;
    const void* src = nullptr;
    size_t size = 0;
    switch (which) {
        case MXA2A_WS_RING: src = p->ring; size = p->ring_bytes; break;
        case MXA2A_WS_SFA: src = p->sfa; size = p->sfa_bytes; break;
        case MXA2A_WS_SFB: src = p->sfb; size = p->sfb_bytes; break;
        case MXA2A_WS_FLAGS: src = p->flags; size = p->flags_bytes; break;
        case MXA2A_WS_APACKED: src = p->a_packed; size = p->apacked_bytes; break;
        default: return MXA2A_ERR_INVALID_OPTION;
    }
    if (bytes_out) *bytes_out = size;
    if (!dst || bytes == 0) return MXA2A_OK;
    int rc = check_device(p);
    if (rc) return rc;
    return cudaMemcpy(dst, src, std::min(bytes, size), cudaMemcpyDeviceToHost) == cudaSuccess ? MXA2A_OK
                                                                                             : MXA2A_ERR_CUDA;
}

int mxa2a_l2_flush(void* buf, size_t bytes, void* stream) {
    if (!buf) return MXA2A_ERR_NULL_PTR;
    if (bytes % 16 || !aligned(buf, 16)) return MXA2A_ERR_MISALIGNED;
    return launch_l2_flush(buf, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MXA2A_OK
                                                                                        : MXA2A_ERR_CUDA;
}

void mxa2a_destroy(mxa2a_plan* p) {
    if (!p) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != p->device) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    if (p->ws) cudaFree(p->ws);
    if (p->split_ws) cudaFree(p->split_ws);
    if (p->io) cudaFree(p->io);
    if (p->rs_scratch) cudaFree(p->rs_scratch);
    for (int i = 0; i < p->ev_count; ++i) {
        cudaEventDestroy(p->ev0[i]);
        cudaEventDestroy(p->ev1[i]);
    }
    delete[] p->ev0;
    delete[] p->ev1;
    if (prev >= 0 && prev != p->device) cudaSetDevice(prev);
    delete p;
}

const char* mxa2a_strerror(int code) {
    switch (code) {
        case MXA2A_OK: return "ok";
        case MXA2A_ERR_INVALID_SHAPE: return "invalid shape";
        case MXA2A_ERR_NULL_PTR: return "null pointer";
        case MXA2A_ERR_MISALIGNED: return "misaligned pointer";
        case MXA2A_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case MXA2A_ERR_CUDA: return "CUDA call failed";
        case MXA2A_ERR_TIMEOUT: return "device wait timed out";
        case MXA2A_ERR_INVALID_OPTION: return "invalid option";
        case MXA2A_ERR_DEVICE_CHECK: return "device consistency check failed";
        case MXA2A_ERR_WRONG_DEVICE: return "current device differs from the plan's device";
        case MXA2A_ERR_SCRATCH_TOO_SMALL: return "problem needs more scratch than the allocation-free entry point holds";
        case MXA2A_ERR_CAPTURE_SPLIT: return "a K-split run cannot be captured into a CUDA graph";
        default: return "unknown error";
    }
}

}  // extern "C"

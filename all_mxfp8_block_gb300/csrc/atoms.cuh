// Packing E8M0 scales into the MMA's scale-factor atoms, one warp task at a
// time (device helper shared by the GEMM kernel's prologue and the pack
// kernels).
//
// Atom layout: for every 128-wide K block kbg and every group g of 128 rows
// (of A) or columns (of B), 512 bytes in which the 4 E8M0 bytes of row x (one
// per 32-wide K sub-block, in K order) form the 32-bit word at index
// (x % 32) * 4 + (x % 128) / 32.
//
// A warp task covers one group g and four consecutive K blocks 4q..4q+3.
// Lane l handles the rows x_j = 128 g + 32 j + l (j = 0..3): the word it
// stores for K block kbg at index l * 4 + j is that row's, so the lane writes
// one 16-byte vector per K block and the warp 512 contiguous bytes, while the
// four words it loads per row are adjacent in the source (one sector).
#pragma once
#include <cstdint>

#include "kernels.cuh"

namespace mxa2a {

// load(kbg, x): the 32-bit scale word of row x for K block kbg (x < nrows).
template <typename LoadWord>
__device__ __forceinline__ void pack_atom_task(uint32_t* atoms, int groups, int kbs, int nrows, int g, int q, int lane,
                                               LoadWord load) {
    // all 16 loads first, from clamped (always valid) coordinates, so that
    // they are in flight together; out-of-range words are zeroed afterwards
    uint32_t w[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int x = min(g * 128 + j * 32 + lane, nrows - 1);
#pragma unroll
        for (int t = 0; t < 4; ++t) w[j][t] = load(min(q * 4 + t, kbs - 1), x);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool row_ok = g * 128 + j * 32 + lane < nrows;
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (!row_ok || q * 4 + t >= kbs) w[j][t] = 0u;
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int kbg = q * 4 + t;
        if (kbg < kbs)
            *reinterpret_cast<uint4*>(atoms + ((size_t)kbg * groups + g) * (kSfAtomBytes / 4) + (size_t)lane * 4) =
                make_uint4(w[0][t], w[1][t], w[2][t], w[3][t]);
    }
}

// Tasks (group g, K-block quad q) of an atom array: groups * ceil(kbs / 4).
__host__ __device__ inline long long atom_tasks(int groups, int kbs) { return (long long)groups * ((kbs + 3) / 4); }

// A CTA-wide pack task through shared memory: group g, K blocks kb0 ..
// kb0 + nkb - 1 (nkb <= kTileKb).  The source rows are read along K (each
// row's nkb words contiguous, consecutive threads on consecutive words: whole
// sectors), the tile is transposed in shared memory (rows kTileKb + 1 words
// apart: conflict-free both ways) and every atom is written as 32 16-byte
// vectors.  tile holds 128 * (kTileKb + 1) words; sync() is a barrier over
// the nthreads taking part, which the call begins and ends with.
constexpr int kTileKb = 16;   // small tasks: most CTAs take part (a task is one round of loads)
constexpr int kTileWords = 128 * (kTileKb + 1);
template <typename LoadWord, typename Sync>
__device__ __forceinline__ void pack_atom_tile(uint32_t* atoms, int groups, int nrows, int g, int kb0, int nkb,
                                               uint32_t* tile, int tid, int nthreads, LoadWord load, Sync sync) {
    constexpr int ld = kTileKb + 1;
    sync();   // the tile's previous contents have been written out
    const int words = 128 * nkb;
    constexpr int U = 8;   // loads in flight per thread
    for (int e0 = tid; e0 < words; e0 += U * nthreads) {
        uint32_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = min(e0 + u * nthreads, words - 1);
            const int i = e / nkb, w = e - (e / nkb) * nkb;
            v[u] = load(kb0 + w, min(g * 128 + i, nrows - 1));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * nthreads;
            if (e < words) {
                const int i = e / nkb, w = e - (e / nkb) * nkb;
                tile[i * ld + w] = g * 128 + i < nrows ? v[u] : 0u;
            }
        }
    }
    sync();
    // atom kb0 + w: lane slot l (32 per atom) writes rows 32 j + l, j = 0..3
    for (int e = tid; e < nkb * 32; e += nthreads) {
        const int w = e >> 5, l = e & 31;
        *reinterpret_cast<uint4*>(atoms + ((size_t)(kb0 + w) * groups + g) * (kSfAtomBytes / 4) + (size_t)l * 4) =
            make_uint4(tile[l * ld + w], tile[(32 + l) * ld + w], tile[(64 + l) * ld + w], tile[(96 + l) * ld + w]);
    }
}
__host__ __device__ inline long long atom_tile_tasks(int groups, int kbs) {
    return (long long)groups * ((kbs + kTileKb - 1) / kTileKb);
}

}  // namespace mxa2a

// Memory-bound helper kernels of libmxa2a: scale-factor packing, the unfused
// pack of A and the benchmark's L2 flush.
//
// Scale-factor "atom" layout used by the MMA: for every 128-wide K block and
// every group of 128 rows (of A) or columns (of B), 512 bytes in which the 4
// E8M0 bytes of row/column x (one per 32-wide K sub-block, in K order) sit as
// one 32-bit word at word index (x % 32) * 4 + (x % 128) / 32.  Copied to TMEM
// with tcgen05.cp 32x128b.warpx4, word (x%32)*4 + c lands in column c of lane
// x%32 (of every lane quarter), which is where the block-scaled MMA reads the
// scale of row/column 32c + x%32.  The pages' scale operands are the E8M0
// tensors scaleA / scaleB (all_to_all_matmul_impl.h, LayoutScaleA/B with byte
// pairs SCALE_C0 = 2): the same bytes in the hardware's own order.
#include <cuda_bf16.h>

#include "atoms.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa2a {

// B_scale [N][K/32] -> atoms [K/128][Ng2][512]; columns N..Ng2*128 get 0.
// One CTA per task of 128 columns x up to kTileKb K blocks, transposed in
// shared memory (atoms.cuh).
__global__ void pack_sfb_kernel(const uint8_t* __restrict__ B_scale, int N, int K, int Ng2, uint32_t* __restrict__ sfb) {
    extern __shared__ uint32_t tile[];
    const int kbs = K / BK;
    const long long tasks = atom_tile_tasks(Ng2, kbs);
    const size_t ld = (size_t)(K / 32);
    auto load = [&](int kbg, int n) { return ptx::ld_nc_u32(B_scale + (size_t)n * ld + (size_t)kbg * 4); };
    for (long long t = blockIdx.x; t < tasks; t += gridDim.x) {
        const int g = (int)(t % Ng2), kb0 = (int)(t / Ng2) * kTileKb;
        pack_atom_tile(sfb, Ng2, N, g, kb0, min(kTileKb, kbs - kb0), tile, threadIdx.x, blockDim.x, load,
                       [] { __syncthreads(); });
    }
}

// Unfused variant: A_packed[m][r*ka + k] = A_seg[r][m][k] (the segments
// concatenated along K; for the all-gather the row blocks stacked along M),
// and the A scales into atoms [K/128][Mg][512].
__global__ void pack_a_kernel(const __grid_constant__ GemmParams p, uint8_t* __restrict__ a_packed) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const int v_per_row = p.K / 16;
    const long long nvec = (long long)p.M * v_per_row;
    for (long long i = tid; i < nvec; i += stride) {
        const int m = (int)(i / v_per_row);
        const int k = (int)(i - (long long)m * v_per_row) * 16;
        const int r = k / p.ka;
        const int kin = k - r * p.ka;
        const SegRow src = seg_row(p, r, m);
        const uint4 v = ptx::ld_nc_v4(p.A_seg[src.seg] + (size_t)src.row * seg_ld(p) + seg_col0(p, r) + kin);
        *reinterpret_cast<uint4*>(a_packed + (size_t)m * p.K + k) = v;
    }
    // the scales: one warp per task of 128 rows x 4 K blocks (atoms.cuh)
    const int kbs = p.K / BK;
    const long long tasks = atom_tasks(p.Mg, kbs);
    uint32_t* sfa = reinterpret_cast<uint32_t*>(p.sfa_stage);
    const int lane = threadIdx.x & 31;
    auto load = [&](int kbg, int m) {
        const int r = kbg / p.kb_per_seg;
        const int kb = kbg - r * p.kb_per_seg;
        const SegRow src = seg_row(p, r, m);
        return ptx::ld_nc_u32(p.A_sf_seg[src.seg] + (size_t)src.row * (seg_ld(p) / 32) + seg_col0(p, r) / 32 +
                              (size_t)kb * 4);
    };
    for (long long t = tid >> 5; t < tasks; t += stride >> 5)
        pack_atom_task(sfa, p.Mg, kbs, p.M, (int)(t % p.Mg), (int)(t / p.Mg), lane, load);
}

__global__ void l2_flush_kernel(uint4* buf, long long n16) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n16;
         i += (long long)gridDim.x * blockDim.x) {
        uint4 v = buf[i];
        v.x += 1u;
        buf[i] = v;
    }
}

static int grid_for(long long work, int threads) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long g = (work + threads - 1) / threads;
    const long long cap = (long long)sms * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

cudaError_t launch_pack_sfb(const uint8_t* B_scale, int N, int K, int Ng2, uint8_t* sfb, cudaStream_t stream) {
    // one CTA per task (at most 8 per SM at a time)
    const long long tasks = atom_tile_tasks(Ng2, K / BK);
    const size_t smem = (size_t)kTileWords * 4;
    pack_sfb_kernel<<<grid_for(tasks * 256, 256), 256, smem, stream>>>(B_scale, N, K, Ng2,
                                                                      reinterpret_cast<uint32_t*>(sfb));
    return cudaGetLastError();
}

cudaError_t launch_pack_a(const GemmParams& p, uint8_t* a_packed, int grid, cudaStream_t stream) {
    const long long work = (long long)p.M * p.K / 16;
    pack_a_kernel<<<grid > 0 ? grid : grid_for(work, 256), 256, 0, stream>>>(p, a_packed);
    return cudaGetLastError();
}

// The collective step of the unfused GEMM + ReduceScatter: one thread per 8
// columns (16 bytes) of a row of P.  Same arithmetic as the fused epilogue:
// fp32 adds of the BF16 partials in rank order from 0, one rounding to BF16.
__global__ void rs_reduce_kernel(const __grid_constant__ RsArgs a) {
    const int vpr = a.N / 8;
    const long long total = (long long)a.nblk * a.rows * vpr;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(i % vpr);
        const long long row = i / vpr;
        const int j = (int)(row / a.rows);
        const size_t off = (size_t)(row - (long long)j * a.rows) * a.N + (size_t)v * 8;
        const uint16_t* own = a.P + (size_t)row * a.N + (size_t)v * 8;
        if (j != a.own) {
            *reinterpret_cast<uint4*>(a.send[j] + off) = ptx::ld_nc_v4(own);
            continue;
        }
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        for (int q = 0; q < a.R; ++q) {
            const uint4 t = ptx::ld_nc_v4(q == a.rank ? own : a.recv[q] + off);
            const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += __uint_as_float(w[e] << 16);
                acc[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
            o[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(a.out + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

cudaError_t launch_rs_reduce(const RsArgs& a, cudaStream_t stream) {
    const long long work = (long long)a.nblk * a.rows * (a.N / 8);
    rs_reduce_kernel<<<grid_for(work, 256), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

// Several copies in one launch, by the SMs (blockIdx.y = the copy): each a
// run of 16-byte vectors between memory the device can address (device
// memory, or pinned host memory through its device address).
struct CopyList {
    static constexpr int kMax = 160;
    int n;
    const uint4* src[kMax];
    uint4* dst[kMax];
    long long n16[kMax];
};

__global__ void copy_list_kernel(const __grid_constant__ CopyList l) {
    const int c = blockIdx.y;
    const uint4* __restrict__ s = l.src[c];
    uint4* __restrict__ d = l.dst[c];
    const long long n = l.n16[c];
    constexpr int U = 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * stride < n) v[u] = s[i + u * stride];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * stride < n) d[i + u * stride] = v[u];
    }
}

// n copies (n <= 160; addresses 16-byte aligned, sizes multiples of 16)
cudaError_t launch_copy_list(int n, const void* const* src, void* const* dst, const size_t* bytes,
                             cudaStream_t stream) {
    CopyList l;
    l.n = n;
    long long biggest = 0;
    for (int i = 0; i < n; ++i) {
        l.src[i] = static_cast<const uint4*>(src[i]);
        l.dst[i] = static_cast<uint4*>(dst[i]);
        l.n16[i] = (long long)(bytes[i] / 16);
        biggest = l.n16[i] > biggest ? l.n16[i] : biggest;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (biggest + 256 * 4 - 1) / (256 * 4);
    const int gx = (int)(want < 1 ? 1 : (want > 8LL * sms ? 8LL * sms : want));
    copy_list_kernel<<<dim3(gx, n), 256, 0, stream>>>(l);
    return cudaGetLastError();
}

cudaError_t launch_l2_flush(void* buf, size_t bytes, cudaStream_t stream) {
    const long long n16 = (long long)(bytes / 16);
    l2_flush_kernel<<<grid_for(n16, 256), 256, 0, stream>>>(reinterpret_cast<uint4*>(buf), n16);
    return cudaGetLastError();
}

}  // namespace mxa2a

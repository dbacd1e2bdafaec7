// mxa2a_run_noalloc: the fused AllToAll + MXFP8 GEMM without any device
// allocation.  The staging ring, the scale-factor tiles, the credit counters
// and the status block live in one file-scope static device array instead of
// a plan's cudaMalloc'd workspace.
//
// For callers that cannot allocate device memory: a runtime whose device
// memory is entirely budgeted by its own pool allocator (a library's
// cudaMalloc there can fail or fragment the pool), or a latency-critical loop
// in which cudaMalloc / cudaFree would implicitly synchronise the device.
//
// Limits and caveats (also stated in include/mxa2a.h):
//  * the scratch array is kNoAllocScratchBytes (16 MiB) and is held by every
//    GPU that loads this library until the process exits;
//  * problems whose staging ring + scale tiles + counters exceed it are
//    rejected with MXA2A_ERR_SCRATCH_TOO_SMALL before any device work;
//  * all calls share the array: calls that overlap on the GPU (two streams,
//    or two host threads) race and corrupt each other's results;
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress), so make that first call before any stream
//    capture begins;
//  * K is never split (no partial-sum buffer), and device-side wait time-outs
//    are not reported: use a plan (mxa2a_run + mxa2a_get_status) for that.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mxa2a.h"
#include "kernels.cuh"

using namespace mxa2a;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// Every byte the allocation-free path uses on the device.  Zero at module load.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(int dev, uint8_t** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
    return cudaSuccess;
}

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

// C: bf16 [M][N], box 32 rows x 32 columns, 64-byte swizzle (the epilogue's TMA stores)
bool encode_c(CUtensorMap* map, void* C, uint64_t M, uint64_t N) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {N, M};
    cuuint64_t strides[1] = {N * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Byte offsets of the regions inside the scratch array for one shape.
struct ScratchLayout {
    size_t flags, status, sfb, sfa, ring, total;
    size_t flags_bytes, sfa_bytes;
};

ScratchLayout layout_for(int R, int64_t M, int64_t ka, int64_t N, int64_t cm, int bn) {
    const int64_t K = (int64_t)R * ka;
    const int64_t Mg = (M + BM - 1) / BM;
    const int64_t Ng2 = 2 * ((N + BN - 1) / BN);
    ScratchLayout L;
    L.flags_bytes = FlagLayout::words(bn, R) * sizeof(unsigned long long);
    L.sfa_bytes = (size_t)(K / BK) * Mg * kSfAtomBytes;
    size_t off = 0;
    L.flags = off; off = align_up(off + L.flags_bytes, 1024);
    L.status = off; off = align_up(off + sizeof(DevStatus), 1024);
    L.sfb = off; off = align_up(off + (size_t)(K / BK) * Ng2 * kSfAtomBytes, 1024);
    L.sfa = off; off = align_up(off + L.sfa_bytes, 1024);
    L.ring = off; off = align_up(off + (size_t)bn * R * cm * ka, 1024);
    L.total = off;
    return L;
}

}  // namespace

extern "C" int mxa2a_run_noalloc(int R, int64_t M, int64_t kPerRank, int64_t N, int64_t commMSize,
                                 int buffer_num, const void* const* A_seg, const void* const* A_scale_seg,
                                 const void* B, const void* B_scale, void* C_bf16, void* stream_v) {
    int rc = mxa2a_validate(R, M, kPerRank, N, commMSize, buffer_num);
    if (rc) return rc;
    const ScratchLayout L = layout_for(R, M, kPerRank, N, commMSize, buffer_num);
    if (L.total > kNoAllocScratchBytes) return MXA2A_ERR_SCRATCH_TOO_SMALL;
    if (!A_seg || !A_scale_seg || !B || !B_scale || !C_bf16) return MXA2A_ERR_NULL_PTR;
    for (int r = 0; r < R; ++r) {
        if (!A_seg[r] || !A_scale_seg[r]) return MXA2A_ERR_NULL_PTR;
        if (!aligned(A_seg[r], 16) || !aligned(A_scale_seg[r], 4)) return MXA2A_ERR_MISALIGNED;
    }
    if (!aligned(B, 16) || !aligned(C_bf16, 16) || !aligned(B_scale, 4)) return MXA2A_ERR_MISALIGNED;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MXA2A_ERR_CUDA;
    if (major != 10 || minor != 3) return MXA2A_ERR_UNSUPPORTED_DEVICE;
    uint8_t* scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return MXA2A_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

    // plan: 128x256 tiles, no K split; staging chunks of about 8 KiB (a plan
    // sizes them from the step and the SM count instead; same bits, other timing)
    const int64_t K = (int64_t)R * kPerRank;
    GemmParams g;
    std::memset(&g, 0, sizeof g);
    g.R = R;
    g.M = (int)M;
    g.N = (int)N;
    g.ka = (int)kPerRank;
    g.K = (int)K;
    g.cm = (int)commMSize;
    g.bn = buffer_num;
    g.steps = (int)(M / commMSize);
    g.Mt = (int)((M + BM - 1) / BM);
    g.Nt = (int)((N + BN - 1) / BN);
    g.tile_n = BN;   // the wide tile: one accumulator, 4 pipeline stages
    g.S = 1;
    g.W = g.Mt * g.Nt;
    g.W_dp = g.W;   // no tail split
    g.S_tail = 1;
    g.kb_per_seg = (int)(kPerRank / BK);
    g.Mg = g.Mt;
    g.Ng2 = 2 * g.Nt;
    g.box_m = (commMSize % BM == 0) ? BM : 64;
    g.zigzag = 1;
    g.rotate = 0;
    g.group_m = 1;
    int64_t want = std::max<int64_t>(1, 8192 / kPerRank);
    int rpc = 1;
    for (int64_t d = 1; d <= commMSize; ++d)
        if (commMSize % d == 0 && d <= want) rpc = (int)d;
    g.rows_per_chunk = rpc;
    g.chunks_per_seg = (int)(commMSize / rpc);
    g.n_copy_tasks = g.steps * R * g.chunks_per_seg;
    g.fused = 1;
    g.exchange_only = 0;
    g.fault_skip_step = -1;
    g.sfb = scratch + L.sfb;
    g.sfa = scratch + L.sfa;
    g.sfa_stage = scratch + L.sfa;
    g.ring = scratch + L.ring;
    g.flags = reinterpret_cast<unsigned long long*>(scratch + L.flags);
    g.status = reinterpret_cast<DevStatus*>(scratch + L.status);
    g.C = static_cast<uint16_t*>(C_bf16);
    g.partial = nullptr;
    g.launch_id = 1;   // the status block is cleared before every launch
    g.timeout_ns = 2000000000LL;
    for (int r = 0; r < R; ++r) {
        g.A_seg[r] = static_cast<const uint8_t*>(A_seg[r]);
        g.A_sf_seg[r] = static_cast<const uint8_t*>(A_scale_seg[r]);
    }
    const int grid = std::max(1, std::min(sms, std::max(g.W, g.n_copy_tasks)));

    CUtensorMap tmap_ring, tmap_b, tmap_c;
    if (!encode_2d(&tmap_ring, g.ring, (uint64_t)kPerRank, (uint64_t)buffer_num * R * commMSize,
                   (uint32_t)g.box_m) ||
        !encode_2d(&tmap_b, B, (uint64_t)K, (uint64_t)N, BN) || !encode_c(&tmap_c, C_bf16, (uint64_t)M, (uint64_t)N))
        return MXA2A_ERR_CUDA;

    // What must start at zero: the credit counters and the status block
    // (contiguous at the front), and the scale tiles of rows past M.
    if (cudaMemsetAsync(scratch + L.flags, 0, L.sfb - L.flags, stream) != cudaSuccess) return MXA2A_ERR_CUDA;
    if (M % BM && cudaMemsetAsync(scratch + L.sfa, 0, L.sfa_bytes, stream) != cudaSuccess) return MXA2A_ERR_CUDA;
    if (launch_pack_sfb(static_cast<const uint8_t*>(B_scale), (int)N, (int)K, g.Ng2, scratch + L.sfb, stream) !=
        cudaSuccess)
        return MXA2A_ERR_CUDA;
    if (launch_mxgemm(g, tmap_ring, tmap_b, tmap_c, grid, true, stream) != cudaSuccess) return MXA2A_ERR_CUDA;
    return MXA2A_OK;
}

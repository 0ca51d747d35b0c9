// bsfp8_api.cu -- host side of the C ABI declared in include/bsfp8.h:
// argument validation, TMA descriptor encoding, per-device set-up, launches
// and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "bsfp8.h"
#include "gemm_kernel.cuh"
#include "quant_kernel.cuh"

namespace bsfp8 {
namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceState {
    bool ready = false;
    int error = FP8_OK;          // sticky set-up failure (e.g. wrong architecture)
    int sm_count = 0;
    uint32_t *status = nullptr;  // 256-byte device allocation, word 0 used
};

std::mutex g_mu;
DeviceState g_dev[MAX_DEVICES];
long long g_wait_limit = -1;     // resolved lazily from the environment
int g_withhold_stage = -1;
unsigned long long *g_trace = nullptr;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

constexpr long long kDefaultWaitLimit = 1ll << 31;

long long wait_limit_locked() {
    if (g_wait_limit < 0) {
        g_wait_limit = kDefaultWaitLimit;
        if (const char *e = std::getenv("BSFP8_WAIT_LIMIT_CYCLES")) {
            long long v = std::atoll(e);
            if (v > 0) g_wait_limit = v;
        }
    }
    return g_wait_limit;
}

template <int BN>
int set_kernel_attrs() {
    if (cudaFuncSetAttribute(bsfp8_gemm_plain<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_plain<BN, SCALE_TOKEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_grouped<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, false, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_grouped_dev<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, false, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN, SCALE_ROWCOL, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN, SCALE_BLOCK32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN, SCALE_BLOCK32, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BN, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    static_assert(smem_bytes<BN, true, false, true>() <= 232448, "shared memory of the per-token pair kernel");
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN, SCALE_TOKEN, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, true, false, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaFuncSetAttribute(bsfp8_gemm_pair<BN, SCALE_TOKEN_E8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BN, true, false, true>()) != cudaSuccess)
        return FP8_ERR_CUDA;
    return FP8_OK;
}

// One-time set-up of the current device.  Returns FP8_OK and fills *out.
int device_setup(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (d.ready) {
        *out = &d;
        return d.error;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (major != 10 || minor != 3) {
        d.ready = true;
        d.error = FP8_ERR_ARCH;
        *out = &d;
        return FP8_ERR_ARCH;
    }
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FP8_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    int rc = set_kernel_attrs<TILE_N>();
    if (rc != FP8_OK) return rc;
    if (!d.status) {
        if (cudaMalloc(&d.status, 256) != cudaSuccess) return FP8_ERR_CUDA;
        // the clear lands before any kernel of a later call, whatever stream
        // that call uses (a memset on the legacy stream is not ordered with a
        // non-blocking stream's work)
        if (cudaMemset(d.status, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return FP8_ERR_CUDA;
    }
    d.sm_count = sms;
    d.ready = true;
    d.error = FP8_OK;
    (void)wait_limit_locked();
    *out = &d;
    return FP8_OK;
}

// 2-D K-major byte tensor [rows, K] with a (BK x box_rows) box, 128-byte swizzle.
int encode_kmajor_raw(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// The same K-major matrix seen as {128 K bytes, rows, K/128 halves}: a box
// {128, box_rows, 2} brings two consecutive 128-K slices of box_rows rows, each
// 128-byte swizzled, one after the other.  Only whole 128-K slices are in the
// view (the third extent rounds down), so a box never reaches past a row.
int encode_kmajor_halves_raw(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
    const int64_t halves = K / BK > 0 ? K / BK : 1;   // a map with K < 128 is never used
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(halves)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(BK)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 2u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// bf16 output C (M x N, row-major) for the epilogue's TMA stores: box of
// STG_COLS columns x BM rows, no swizzle; rows past M are clipped by the TMA.
int encode_out_raw(CUtensorMap *m, void *C, int64_t M, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2u};
    const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(BM)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// E4M3 output codes (M x N bytes, row-major) for the quantized-output
// epilogue: box of 32 bytes x BM rows, no swizzle; rows past M are clipped.
int encode_outq_raw(CUtensorMap *m, void *Cq, int64_t M, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N)};
    const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(BM)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Cq, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// A tensor map is a pure function of its encode arguments, so one cached by
// those arguments stays valid whatever later happens to the memory behind it.
// The cache saves the host ~2 us per map (a grouped call encodes one per group).
struct MapKey {
    int kind;   // 0: 2D K-major, 1: 3D K-major halves, 2: bf16 output, 3: E4M3 output
    int box;
    const void *base;
    int64_t a, b;
    bool operator==(const MapKey &o) const {
        return kind == o.kind && box == o.box && base == o.base && a == o.a && b == o.b;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
        h ^= static_cast<uint64_t>(k.a) + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2);
        h ^= static_cast<uint64_t>(k.b) + 0x85157AF5ull + (h << 6) + (h >> 2);
        h ^= static_cast<uint64_t>(k.kind * 1024 + k.box) + (h << 6) + (h >> 2);
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMaxCachedMaps = 4096;
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

template <typename Encode>
int cached_map(CUtensorMap *m, const MapKey &k, Encode encode) {
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(k);
        if (it != g_maps.end()) {
            *m = it->second;
            return FP8_OK;
        }
    }
    const int rc = encode(m);
    if (rc != FP8_OK) return rc;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
    g_maps.emplace(k, *m);
    return FP8_OK;
}

int encode_kmajor(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
    return cached_map(m, MapKey{0, box_rows, base, rows, K},
                      [&](CUtensorMap *o) { return encode_kmajor_raw(o, base, rows, K, box_rows); });
}
int encode_kmajor_halves(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
    return cached_map(m, MapKey{1, box_rows, base, rows, K},
                      [&](CUtensorMap *o) { return encode_kmajor_halves_raw(o, base, rows, K, box_rows); });
}
int encode_out(CUtensorMap *m, void *C, int64_t M, int64_t N) {
    return cached_map(m, MapKey{2, BM, C, M, N}, [&](CUtensorMap *o) { return encode_out_raw(o, C, M, N); });
}
int encode_outq(CUtensorMap *m, void *Cq, int64_t M, int64_t N) {
    return cached_map(m, MapKey{3, BM, Cq, M, N}, [&](CUtensorMap *o) { return encode_outq_raw(o, Cq, M, N); });
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(int64_t M, int64_t N, int64_t K) {
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (M >= lim || N >= lim || K >= lim) return FP8_ERR_SHAPE;
    if ((N % 32) != 0 || (K % 32) != 0) return FP8_ERR_SHAPE;
    return FP8_OK;
}

int check_mode(int mode) {
    return (mode == FP8_PATH_AUTO || mode == FP8_PATH_NATIVE || mode == FP8_PATH_PROMOTE)
               ? FP8_OK
               : FP8_ERR_MODE;
}

int zero_fill(void *C, int64_t elems, cudaStream_t stream) {
    const int64_t n16 = (elems * 2) / 16;
    const int64_t tail = (elems * 2) % 16;
    if (n16 > 0) {
        int blocks = static_cast<int>(n16 / 256 + 1);
        if (blocks > 4096) blocks = 4096;
        bsfp8_zero_fill<<<blocks, 256, 0, stream>>>(static_cast<uint4 *>(C), n16);
        if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
    }
    if (tail) {   // N % 32 == 0 makes rows 64-byte multiples: no tail can occur
        return FP8_ERR_SHAPE;
    }
    return FP8_OK;
}

void fill_common(Common &c, int64_t M, int64_t N, int64_t K, int mode, DeviceState *d, int BN) {
    std::memset(&c, 0, sizeof c);
    c.M = static_cast<int>(M);
    c.N = static_cast<int>(N);
    c.K = static_cast<int>(K);
    c.KB = static_cast<int>(K / 32);
    c.KS = static_cast<int>((K + BK - 1) / BK);
    c.mt = static_cast<int>((M + BM - 1) / BM);
    c.nt = static_cast<int>((N + BN - 1) / BN);
    c.num_tiles = c.mt * c.nt;
    c.mode = mode;
    c.status = d->status;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        c.wait_limit = wait_limit_locked();
        c.withhold_stage = g_withhold_stage;
        c.trace = g_trace;
    }
}

template <int BN, int SK = SCALE_BLOCK32>
int launch_plain(const void *A, const float *sA, const void *B, const float *sB, void *C,
                 int64_t M, int64_t N, int64_t K, int mode, DeviceState *d, cudaStream_t stream) {
    PlainArgs args;
    std::memset(&args, 0, sizeof args);
    fill_common(args.c, M, N, K, mode, d, BN);
    int rc = encode_kmajor(&args.tmA, A, M, K, BM);
    if (rc != FP8_OK) return rc;
    rc = encode_kmajor(&args.tmB, B, N, K, BN);
    if (rc != FP8_OK) return rc;
    rc = encode_out(&args.tmC, C, M, N);
    if (rc != FP8_OK) return rc;
    args.e.A = static_cast<const uint8_t *>(A);
    args.e.sA = sA;
    args.e.sB = sB;
    args.e.C = static_cast<__nv_bfloat16 *>(C);
    int grid = args.c.num_tiles < d->sm_count ? args.c.num_tiles : d->sm_count;
    bsfp8_gemm_plain<BN, SK><<<grid, NUM_THREADS, smem_bytes<BN>(), stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// CTA-pair launch: 256-row tiles, each CTA of a pair loads 128 rows of A and
// 128 of B's 256 columns; the grid is a whole number of pairs.
template <int BN, int SK = SCALE_BLOCK32, bool RES = false, bool QOUT = false>
int launch_pair(const void *A, const float *sA, const void *B, const float *sB, void *C,
                int64_t M, int64_t N, int64_t K, int mode, DeviceState *d, cudaStream_t stream,
                const void *R = nullptr, float *sC = nullptr) {
    PlainArgs args;
    std::memset(&args, 0, sizeof args);
    fill_common(args.c, M, N, K, mode, d, BN);
    args.c.mt = static_cast<int>((M + 2 * BM - 1) / (2 * BM));
    args.c.num_tiles = args.c.mt * args.c.nt;
    int rc = encode_kmajor(&args.tmA, A, M, K, BM);
    if (rc != FP8_OK) return rc;
    rc = encode_kmajor(&args.tmB, B, N, K, BN / 2);
    if (rc != FP8_OK) return rc;
    if constexpr (QOUT) {   // C holds the E4M3 codes
        rc = encode_outq(&args.tmQ, C, M, N);
        args.Cq = static_cast<uint8_t *>(C);
        args.sC = sC;
    } else {
        rc = encode_out(&args.tmC, C, M, N);
    }
    if (rc != FP8_OK) return rc;
    rc = encode_kmajor_halves(&args.tmA3, A, M, K, BM);
    if (rc != FP8_OK) return rc;
    rc = encode_kmajor_halves(&args.tmB3, B, N, K, BN / 2);
    if (rc != FP8_OK) return rc;
    args.e.A = static_cast<const uint8_t *>(A);
    args.e.sA = sA;
    args.e.sB = sB;
    args.e.C = static_cast<__nv_bfloat16 *>(C);
    if constexpr (RES) {
        args.R = static_cast<const __nv_bfloat16 *>(R);
        rc = encode_out(&args.tmR, const_cast<void *>(R), M, N);
        if (rc != FP8_OK) return rc;
    }
    const int pairs = args.c.num_tiles < d->sm_count / 2 ? args.c.num_tiles : d->sm_count / 2;
    constexpr bool ROWA = SK == SCALE_TOKEN || SK == SCALE_TOKEN_E8;   // per-row A scale lines
    bsfp8_gemm_pair<BN, SK, RES, QOUT><<<2 * pairs, NUM_THREADS, smem_bytes<BN, true, false, ROWA>(), stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int BN>
int launch_grouped(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K,
                   int32_t G, int mode, DeviceState *d, cudaStream_t stream) {
    static_assert(sizeof(GroupedArgs) < 32000, "kernel parameter space");
    GroupedArgs *args = new GroupedArgs;   // large: keep it off the stack
    std::memset(args, 0, sizeof *args);
    fill_common(args->c, 0, N, K, mode, d, BN);
    args->c.G = G;
    args->c.Ms = Ms;
    for (int g = 0; g < G; ++g) {
        // rows are only bounded by the tensor map; the kernel never requests
        // B rows beyond N, so the map's row count is exactly N.
        int rc = encode_kmajor(&args->tmB[g], groups[g].B, N, K, BN);
        if (rc != FP8_OK) {
            delete args;
            return rc;
        }
        args->e[g].A = static_cast<const uint8_t *>(groups[g].A);
        args->e[g].sA = groups[g].sA;
        args->e[g].sB = groups[g].sB;
        args->e[g].C = static_cast<__nv_bfloat16 *>(groups[g].C);
    }
    bsfp8_gemm_grouped<BN><<<d->sm_count, NUM_THREADS, smem_bytes<BN, false, true>(), stream>>>(*args);
    delete args;
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// Grouped launch with device-resident records: the prepare kernel builds the
// groups' B tensor maps in the workspace, the GEMM kernel reads maps and
// records from device memory.  Both are ordinary launches on `stream`, so a
// captured graph replays them with whatever the table holds at that time.
constexpr int64_t kMapBytes = 128;
int64_t grouped_ws_bytes(int32_t G) { return static_cast<int64_t>(G) * (kMapBytes + 4) + 256; }

template <int BN>
int launch_grouped_dev(const GroupRecord *table, const int32_t *Ms, int64_t N, int64_t K, int32_t G,
                       CUtensorMap *maps, int32_t *valid, int mode, DeviceState *d, cudaStream_t stream) {
    // the template: shape N x K, box of BN rows; its base (here the map slots'
    // own address, any valid one will do) is replaced per group on the device
    CUtensorMap tmpl;
    int rc = encode_kmajor(&tmpl, maps, N, K, BN);
    if (rc != FP8_OK) return rc;
    bsfp8_grouped_prepare<<<(G + 3) / 4, 128, 0, stream>>>(tmpl, table, G, maps, valid, d->status);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
    GroupedDevArgs args;
    std::memset(&args, 0, sizeof args);
    fill_common(args.c, 0, N, K, mode, d, BN);
    args.c.G = G;
    args.c.Ms = Ms;
    args.table = table;
    args.maps = maps;
    args.valid = valid;
    bsfp8_gemm_grouped_dev<BN><<<d->sm_count, NUM_THREADS, smem_bytes<BN, false, true>(), stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ------------------------------------------- allocation-free entry point ----
// fp8_gemm_blockscaled_noalloc runs the same kernel, but the device status
// word it needs lives in this file-scope array instead of memory obtained from
// cudaMalloc.  Every GPU that loads the library holds these 256 bytes until
// the process exits.  Host code only ever uses the address returned by
// cudaGetSymbolAddress for the current device: the name itself is a host-side
// stand-in, not a device pointer.
constexpr int kNoAllocScratchWords = 64;   // 256 bytes; word 0 is the status word
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

struct NoAllocState {
    bool ready = false;
    int error = FP8_OK;
    int sm_count = 0;
    uint32_t *scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[MAX_DEVICES];

// One-time set-up of the current device for the allocation-free entry point:
// architecture check, kernel attributes, and the device address of the
// static scratch array (cleared once).  Allocates nothing.
int noalloc_setup(NoAllocState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocState &st = g_noalloc[dev];
    if (st.ready) {
        *out = &st;
        return st.error;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (major != 10 || minor != 3) {
        st.ready = true;
        st.error = FP8_ERR_ARCH;
        *out = &st;
        return FP8_ERR_ARCH;
    }
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FP8_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (set_kernel_attrs<TILE_N>() != FP8_OK) return FP8_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return FP8_ERR_CUDA;
    // the status word must start at zero (later calls only OR bits into it),
    // and the clear must land before the first kernel, on whatever stream
    if (cudaMemset(p, 0, sizeof(uint32_t) * kNoAllocScratchWords) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return FP8_ERR_CUDA;
    st.scratch = static_cast<uint32_t *>(p);
    st.sm_count = sms;
    st.ready = true;
    st.error = FP8_OK;
    (void)wait_limit_locked();
    *out = &st;
    return FP8_OK;
}

template <int BN>
int launch_plain_noalloc(const void *A, const float *sA, const void *B, const float *sB, void *C,
                         int64_t M, int64_t N, int64_t K, NoAllocState *st, cudaStream_t stream) {
    PlainArgs args;
    std::memset(&args, 0, sizeof args);
    Common &c = args.c;
    c.M = static_cast<int>(M);
    c.N = static_cast<int>(N);
    c.K = static_cast<int>(K);
    c.KB = static_cast<int>(K / 32);
    c.KS = static_cast<int>((K + BK - 1) / BK);
    c.mt = static_cast<int>((M + BM - 1) / BM);
    c.nt = static_cast<int>((N + BN - 1) / BN);
    c.num_tiles = c.mt * c.nt;
    c.mode = FP8_PATH_AUTO;
    c.status = st->scratch;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        c.wait_limit = wait_limit_locked();
        c.withhold_stage = g_withhold_stage;   // debug control, -1 unless a test sets it
        c.trace = nullptr;
    }
    int rc = encode_kmajor(&args.tmA, A, M, K, BM);
    if (rc != FP8_OK) return rc;
    rc = encode_kmajor(&args.tmB, B, N, K, BN);
    if (rc != FP8_OK) return rc;
    rc = encode_out(&args.tmC, C, M, N);
    if (rc != FP8_OK) return rc;
    args.e.A = static_cast<const uint8_t *>(A);
    args.e.sA = sA;
    args.e.sB = sB;
    args.e.C = static_cast<__nv_bfloat16 *>(C);
    const int grid = c.num_tiles < st->sm_count ? c.num_tiles : st->sm_count;
    bsfp8_gemm_plain<BN><<<grid, NUM_THREADS, smem_bytes<BN>(), stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// Reads and clears one device status word: `stream` has been synchronised;
// the clear is ordered on `stream` and waited for.
int read_and_clear(uint32_t *word_dev, uint32_t *word, cudaStream_t stream) {
    *word = 0;
    if (!word_dev) return FP8_OK;
    if (cudaMemcpy(word, word_dev, sizeof *word, cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
    if (*word != 0 && (cudaMemsetAsync(word_dev, 0, sizeof *word, stream) != cudaSuccess ||
                       cudaStreamSynchronize(stream) != cudaSuccess))
        return FP8_ERR_CUDA;
    return FP8_OK;
}

}  // namespace
}  // namespace bsfp8

using namespace bsfp8;

extern "C" {

int fp8_gemm_blockscaled_ex(const void *A, const float *sA, const void *B, const float *sB,
                            void *C, int64_t M, int64_t N, int64_t K, int mode,
                            cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    rc = check_mode(mode);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C) return FP8_ERR_NULL;
    if (!aligned(C, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return zero_fill(C, M * N, stream);
    // Every tile promotes: the single-CTA kernel, whose promotion pipeline
    // waits on no cross-CTA releases, runs this path faster than CTA pairs.
    if (mode == FP8_PATH_PROMOTE) return launch_plain<TILE_N>(A, sA, B, sB, C, M, N, K, mode, d, stream);
    return launch_pair<TILE_N>(A, sA, B, sB, C, M, N, K, mode, d, stream);
}

int fp8_gemm_blockscaled(const void *A, const float *sA, const void *B, const float *sB, void *C,
                         int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return fp8_gemm_blockscaled_ex(A, sA, B, sB, C, M, N, K, FP8_PATH_AUTO, stream);
}

int fp8_gemm_blockscaled_residual(const void *A, const float *sA, const void *B, const float *sB,
                                  const void *R, void *C, int64_t M, int64_t N, int64_t K,
                                  cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C || !R) return FP8_ERR_NULL;
    if (!aligned(C, 16) || !aligned(R, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) {   // C = R
        if (C == R) return FP8_OK;
        return cudaMemcpyAsync(C, R, static_cast<size_t>(M * N) * 2, cudaMemcpyDeviceToDevice, stream) ==
                       cudaSuccess
                   ? FP8_OK
                   : FP8_ERR_CUDA;
    }
    return launch_pair<TILE_N, SCALE_BLOCK32, true>(A, sA, B, sB, C, M, N, K, FP8_PATH_AUTO, d, stream, R);
}

int fp8_gemm_blockscaled_quant(const void *A, const float *sA, const void *B, const float *sB, void *Cq,
                               float *sC, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!Cq || !sC) return FP8_ERR_NULL;
    if (!aligned(Cq, 16) || !aligned(sC, 4)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) {   // C = 0: every block all zero, so codes 0 and scales 1
        rc = zero_fill(Cq, M * N / 2, stream);
        if (rc != FP8_OK) return rc;
        const int64_t ns = (M + 31) / 32 * (N / 32);
        int blocks = static_cast<int>(ns / 256 + 1);
        if (blocks > 4096) blocks = 4096;
        bsfp8_fill_f32<<<blocks, 256, 0, stream>>>(sC, 1.0f, ns);
        return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
    }
    return launch_pair<TILE_N, SCALE_BLOCK32, false, true>(A, sA, B, sB, Cq, M, N, K, FP8_PATH_AUTO, d, stream,
                                                           nullptr, sC);
}

int fp8_gemm_rowcol(const void *A, const float *sA, const void *B, const float *sB, void *C,
                    int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C) return FP8_ERR_NULL;
    if (!aligned(C, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return zero_fill(C, M * N, stream);
    return launch_pair<TILE_N, SCALE_ROWCOL, false>(A, sA, B, sB, C, M, N, K, FP8_PATH_AUTO, d, stream);
}

int fp8_gemm_pertoken_ex(const void *A, const float *sA, const void *B, const float *sB, void *C,
                         int64_t M, int64_t N, int64_t K, int mode, cudaStream_t stream) {
    int rc = check_mode(mode);
    if (rc != FP8_OK) return rc;
    rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C) return FP8_ERR_NULL;
    if (!aligned(C, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return zero_fill(C, M * N, stream);
    // NATIVE: CTA pairs with per-row UE8M0 scale lines (the scales must be
    // powers of two); otherwise the promotion path on single-CTA tiles (faster
    // for that path than CTA pairs)
    if (mode == FP8_PATH_NATIVE)
        return launch_pair<TILE_N, SCALE_TOKEN, false>(A, sA, B, sB, C, M, N, K, FP8_PATH_NATIVE, d, stream);
    return launch_plain<TILE_N, SCALE_TOKEN>(A, sA, B, sB, C, M, N, K, FP8_PATH_PROMOTE, d, stream);
}

int fp8_gemm_pertoken(const void *A, const float *sA, const void *B, const float *sB, void *C,
                      int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return fp8_gemm_pertoken_ex(A, sA, B, sB, C, M, N, K, FP8_PATH_AUTO, stream);
}

int fp8_gemm_pertoken_e8m0(const void *A, const void *sA, const void *B, const float *sB, void *C,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C) return FP8_ERR_NULL;
    if (!aligned(C, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sB, 4)) return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return zero_fill(C, M * N, stream);
    return launch_pair<TILE_N, SCALE_TOKEN_E8, false>(A, static_cast<const float *>(sA), B, sB, C, M, N, K,
                                                      FP8_PATH_NATIVE, d, stream);
}

int fp8_gemm_blockscaled_noalloc(const void *A, const float *sA, const void *B, const float *sB,
                                 void *C, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_shape(M, N, K);
    if (rc != FP8_OK) return rc;
    if (M == 0 || N == 0) return FP8_OK;
    if (!C) return FP8_ERR_NULL;
    if (!aligned(C, 16)) return FP8_ERR_ALIGN;
    if (K > 0) {
        if (!A || !B || !sA || !sB) return FP8_ERR_NULL;
        if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4))
            return FP8_ERR_ALIGN;
    }
    // the scratch is the fixed 256-byte array above; its size does not grow
    // with M, N or K, so the shape checks above are the only size limits
    static_assert(sizeof(uint32_t) * kNoAllocScratchWords <= FP8_NOALLOC_SCRATCH_BYTES,
                  "scratch larger than the documented maximum");
    NoAllocState *st = nullptr;
    rc = noalloc_setup(&st);
    if (rc != FP8_OK) return rc;
    if (K == 0) return zero_fill(C, M * N, stream);
    return launch_plain_noalloc<TILE_N>(A, sA, B, sB, C, M, N, K, st, stream);
}

int fp8_gemm_grouped_ex(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K,
                        int32_t G, int mode, cudaStream_t stream) {
    int rc = check_shape(0, N, K);
    if (rc != FP8_OK) return rc;
    rc = check_mode(mode);
    if (rc != FP8_OK) return rc;
    if (G < 0) return FP8_ERR_SHAPE;
    if (G == 0 || N == 0) return FP8_OK;
    if (!groups || !Ms) return FP8_ERR_NULL;
    if (!aligned(Ms, 4)) return FP8_ERR_ALIGN;
    for (int g = 0; g < G; ++g) {
        const fp8_group_desc &e = groups[g];
        if (!e.A || !e.B || !e.sA || !e.sB || !e.C) return FP8_ERR_NULL;
        if (!aligned(e.A, 16) || !aligned(e.B, 16) || !aligned(e.C, 16) || !aligned(e.sA, 4) ||
            !aligned(e.sB, 4))
            return FP8_ERR_ALIGN;
    }
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return FP8_ERR_SHAPE;   // row counts are on the device: no host-side zero fill
    for (int32_t g0 = 0; g0 < G; g0 += FP8_MAX_GROUPS_PER_LAUNCH) {
        const int32_t n = (G - g0) < FP8_MAX_GROUPS_PER_LAUNCH ? (G - g0) : FP8_MAX_GROUPS_PER_LAUNCH;
        rc = launch_grouped<TILE_N>(groups + g0, Ms + g0, N, K, n, mode, d, stream);
        if (rc != FP8_OK) return rc;
    }
    return FP8_OK;
}

int fp8_gemm_grouped(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K,
                     int32_t G, cudaStream_t stream) {
    return fp8_gemm_grouped_ex(groups, Ms, N, K, G, FP8_PATH_AUTO, stream);
}

int64_t fp8_grouped_workspace_bytes(int32_t G) { return G < 0 ? 0 : grouped_ws_bytes(G); }

int fp8_gemm_grouped_device(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K, int32_t G,
                            void *workspace, int64_t workspace_bytes, cudaStream_t stream) {
    static_assert(sizeof(fp8_group_desc) == sizeof(GroupRecord), "record layout");
    int rc = check_shape(0, N, K);
    if (rc != FP8_OK) return rc;
    if (G < 0) return FP8_ERR_SHAPE;
    if (G == 0 || N == 0) return FP8_OK;
    if (!groups || !Ms || !workspace) return FP8_ERR_NULL;
    if (!aligned(groups, 8) || !aligned(Ms, 4) || !aligned(workspace, 128)) return FP8_ERR_ALIGN;
    if (workspace_bytes < grouped_ws_bytes(G)) return FP8_ERR_SHAPE;
    DeviceState *d = nullptr;
    rc = device_setup(&d);
    if (rc != FP8_OK) return rc;
    if (K == 0) return FP8_ERR_SHAPE;   // as fp8_gemm_grouped: no host-side zero fill
    CUtensorMap *maps = static_cast<CUtensorMap *>(workspace);
    int32_t *valid = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + static_cast<int64_t>(G) * kMapBytes);
    const GroupRecord *table = reinterpret_cast<const GroupRecord *>(groups);
    for (int32_t g0 = 0; g0 < G; g0 += FP8_MAX_GROUPS_PER_LAUNCH) {
        const int32_t n = (G - g0) < FP8_MAX_GROUPS_PER_LAUNCH ? (G - g0) : FP8_MAX_GROUPS_PER_LAUNCH;
        rc = launch_grouped_dev<TILE_N>(table + g0, Ms + g0, N, K, n, maps + g0, valid + g0, FP8_PATH_AUTO, d, stream);
        if (rc != FP8_OK) return rc;
    }
    return FP8_OK;
}

int fp8_status_query(cudaStream_t stream, int *status) {
    if (!status) return FP8_ERR_NULL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return FP8_ERR_CUDA;
    // the words of whichever entry points have run on this device (the
    // regular status word and word 0 of the allocation-free scratch array);
    // nothing is set up or allocated here
    uint32_t *regular = nullptr, *noalloc = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev[dev].ready) regular = g_dev[dev].status;
        if (g_noalloc[dev].ready) noalloc = g_noalloc[dev].scratch;
    }
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
    uint32_t w1 = 0, w2 = 0;
    int rc = read_and_clear(regular, &w1, stream);
    if (rc != FP8_OK) return rc;
    rc = read_and_clear(noalloc, &w2, stream);
    if (rc != FP8_OK) return rc;
    const uint32_t word = w1 | w2;
    *status = (word & STATUS_TIMEOUT)  ? FP8_ERR_TIMEOUT
              : (word & STATUS_RECORD) ? FP8_ERR_RECORD
              : (word & STATUS_SCALE)  ? FP8_ERR_SCALE
                                       : FP8_OK;
    return FP8_OK;
}

const char *fp8_strerror(int code) {
    switch (code) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_NULL: return "FP8_ERR_NULL: a required pointer is NULL";
        case FP8_ERR_SHAPE: return "FP8_ERR_SHAPE: bad size (negative, N or K not a multiple of 32, >= 2^31, or G)";
        case FP8_ERR_ALIGN: return "FP8_ERR_ALIGN: A/B/C must be 16-byte and sA/sB 4-byte aligned";
        case FP8_ERR_ARCH: return "FP8_ERR_ARCH: the current device is not sm_103";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA: a CUDA call failed";
        case FP8_ERR_MODE: return "FP8_ERR_MODE: unknown path mode or debug key";
        case FP8_ERR_SCALE: return "FP8_ERR_SCALE: native path forced with a scale that is not a power of two";
        case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT: a device-side wait ran out";
        case FP8_ERR_RECORD: return "FP8_ERR_RECORD: a device-resident group record held a null or misaligned pointer (group skipped)";
        default: return "unknown FP8 status code";
    }
}

int fp8_version(void) { return BSFP8_VERSION; }

int fp8_debug_set(int key, int64_t value) {
    std::lock_guard<std::mutex> lk(g_mu);
    switch (key) {
        case FP8_DEBUG_WAIT_LIMIT_CYCLES:
            g_wait_limit = value > 0 ? value : kDefaultWaitLimit;
            return FP8_OK;
        case FP8_DEBUG_WITHHOLD_STAGE:
            g_withhold_stage = value >= 0 ? static_cast<int>(value) : -1;
            return FP8_OK;
        case FP8_DEBUG_TRACE_BUFFER:
            g_trace = reinterpret_cast<unsigned long long *>(static_cast<uintptr_t>(value));
            return FP8_OK;
        default:
            return FP8_ERR_MODE;
    }
}

int fp8_quantize_blocks(const void *x, void *q, float *s, int64_t M, int64_t K, cudaStream_t stream) {
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || K < 0 || M >= lim || K >= lim || (K % 32) != 0) return FP8_ERR_SHAPE;
    if (M == 0 || K == 0) return FP8_OK;
    if (!x || !q || !s) return FP8_ERR_NULL;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return FP8_ERR_ALIGN;
    DeviceState *d = nullptr;
    const int rc = device_setup(&d);   // architecture check (sm_103 only)
    if (rc != FP8_OK) return rc;
    const int64_t MB = (M + 31) / 32;
    const dim3 grid(static_cast<unsigned>((K + QT_COLS - 1) / QT_COLS),
                    static_cast<unsigned>(MB < 65535 ? MB : 65535));
    bsfp8_quantize_blocks<<<grid, QT_THREADS, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x),
                                                          static_cast<uint8_t *>(q), s, M, K);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

void fp8_lib_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < MAX_DEVICES; ++i) {
        if (g_dev[i].status) {
            int cur = 0;
            if (cudaGetDevice(&cur) == cudaSuccess && cudaSetDevice(i) == cudaSuccess) {
                cudaFree(g_dev[i].status);
                cudaSetDevice(cur);
            }
        }
        g_dev[i] = DeviceState();
        // the allocation-free entry point's static array stays (it belongs to
        // the loaded module); its set-up runs again on the next call
        g_noalloc[i] = NoAllocState();
    }
    std::lock_guard<std::mutex> lm(g_map_mu);
    g_maps.clear();
}

}  // extern "C"

// gemm_kernel.cuh -- persistent, warp-specialised block-scaled E4M3 GEMM for
// sm_103a (tcgen05 tensor cores, tensor-memory accumulators, TMA).
//
// Computes C[m,n] = bf16( sum_kb sA[m/32][kb] * sB[n/32][kb] * sum_{k in kb}
// A[m,k] B[n,k] ) (FP8 GEMM library article, hncyxsy.com/news/241433,
// sections 2.2-2.3: 32x32 block scales that take part in the accumulation),
// for one problem or for a group of independent problems (same article,
// section 4.2: one launch, each block looks up its problem in a table).
//
// Kernels (one body, gemm_body):
//   bsfp8_gemm_pair     single problems on CTA pairs (cta_group::2): 256 x 256
//                       output tiles, one M=256/N=256/K=32 MMA per 32-K block
//                       issued by the pair's leader; operand stages of 256 K
//                       arrive as one 3D TMA box per operand; template
//                       variants for per-row/column scales, per-token A
//                       scales (fp32 or UE8M0 bytes), a fused residual add
//                       and an output quantized to E4M3 with 32x32 scales
//   bsfp8_gemm_plain    single problems, one CTA per 128 x 256 tile (the
//                       allocation-free entry point, and the promotion path
//                       when the caller pins it: with no cross-CTA releases
//                       per 32-K partial it runs that path faster)
//   bsfp8_gemm_grouped  many decode problems in one launch: 64-row tiles, A
//                       rows by cp.async (their count lives on the device)
// An M=128 MMA costs ~116 cycles for any N <= 128 but only ~160 for N = 256,
// so N = 256 is what reaches the tensor peak.  The MMA issue blocks until the
// pipe accepts the next MMA (it holds about one), so the issuing thread does
// as little as possible between MMAs, and no warp of its sub-partition polls
// or computes while it issues (two busy neighbours halve its issue rate).
//
// Roles (384 threads, one CTA per SM, persistent over output tiles; in a pair
// each CTA runs every role on its half: both CTAs' operand loads complete on
// the leader's barriers (cta_group::2 TMA), and the peer's MMA warp forwards
// the readiness of its scale lines with relaxed cluster-scope arrives):
//   warp 0     producer: TMA loads of the A and B K-slices into a ring of
//              shared-memory stages (128-byte swizzle; grouped problems: A
//              rows by cp.async).
//   warp 1     MMA issuer, run by lane 0 alone.  Native path: it copies a
//              stage's UE8M0 scale lines into tensor memory (tcgen05.cp) and
//              issues its kind::mxf8f6f4 block-scaled MMAs back to back as one
//              straight line, testing the next stage's barriers inside the asm
//              block of the last two.  Promotion path: one unscaled
//              kind::f8f6f4 MMA and one commit per 32-K block into one of two
//              tensor-memory partials (partials as wide as tensor memory
//              allows); a stage's scale entry is released once the epilogue
//              has read all of its partials.
//   warp 2     path verdict: scans each tile's scales ahead of time and decides
//              native (all positive normal powers of two) or promotion; the
//              first tile's scan is shared by warps 1, 2 and 4-11 at start.
//              With per-token native scales it builds the per-row scale lines
//              instead.
//   warp 3     scale warp: cp.async of each stage's fp32 scales into a ring
//              that runs ahead of the operand ring, then the UE8M0 lines (8
//              identical 16-byte lines per 128 rows, read four times by
//              tcgen05.cp) that the MMA warp copies into tensor memory.
//   warps 4-11 epilogue: native tiles drain the accumulator into registers
//              (one warp per column half polls for it; the others wait in the
//              half's named barrier), release it to the MMA thread at once,
//              then convert to bf16 (or to E4M3 codes and block scales) and
//              write 128 x 32 chunks through a shared-memory staging buffer
//              with TMA stores (grouped tiles: 16-byte stores); promotion
//              tiles accumulate acc += (sA*sB) * partial per 32-K block in fp32
//              registers, with sA and sB read from the stage's scale entry,
//              and store at the end.
//
// The K loop of every tile runs whole and in ascending K order, with a tile
// shape that depends only on the kernel, never on M: no split-K, no stream-K,
// so each output row is independent of M and of the other rows ("AI Infra
// 进阶：如何让大模型输出确定的结果", aif.amtbbs.org post 29992, section 1).
//
// Tensor memory (512 columns): accumulator / partial 0 at [0, BN), partial 1
// at [BN, 2 BN), the per-stage scale columns at [SF_COL0, ...).  For BN = 256
// the scale columns share partial 1's range; path changes between tiles wait
// for both buffers to drain first.
//
// Every wait is bounded (clock64 budget).  On expiry a CTA-wide abort flag
// and the device status word are set, every role leaves its loop, in-flight
// TMA loads and MMAs are drained with bounded waits, tensor memory is freed
// and the kernel returns.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"
#include "quant_kernel.cuh"

namespace bsfp8 {

constexpr int BM = 128;            // rows of A per tile (MMA M)
constexpr int BK = 128;            // K elements (= bytes) per pipeline stage
constexpr int KB_PER_STAGE = 4;    // 32-K scale blocks per stage
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int MAX_GROUPS = 64;
constexpr int GROUP_M = 8;         // tile-order swizzle width (m-tiles) for L2 reuse
constexpr int TILE_N = 256;        // the BN every launch uses

enum : uint32_t { STATUS_TIMEOUT = 1u, STATUS_SCALE = 2u, STATUS_RECORD = 4u };
enum : int { PATH_AUTO = 0, PATH_NATIVE = 1, PATH_PROMOTE = 2 };
// Scale layouts (a kernel template parameter, so each layout compiles its own
// kernel and the block-scaled kernels carry no code for the others):
// SCALE_BLOCK32: sA [ceil(M/32)][K/32], sB [N/32][K/32] block scales.
// SCALE_ROWCOL: sA [M] and sB [N], constant along K: the MMAs run with unit
// scales and the epilogue multiplies each output by sA[m] * sB[n].
// SCALE_TOKEN: sA [M][K/32] fp32, one scale per row of A per 32-K block (per
// token), sB [N/32][K/32] blocks: single CTAs take the promotion path (the
// epilogue thread of row m reads sA[m][kb] itself), CTA pairs the native path
// with per-row scale lines built by warp 2.
// SCALE_TOKEN_E8: the same with sA as UE8M0 bytes (2^(e-127)): CTA pairs only,
// native path; warp 2 copies the bytes into the lines without converting them.
enum : int { SCALE_BLOCK32 = 0, SCALE_ROWCOL = 1, SCALE_TOKEN = 2, SCALE_TOKEN_E8 = 3 };

template <int BN_, bool PAIR_ = false, bool GROUPED_ = false, bool ROWA_ = false>
struct Cfg {
    static constexpr int BN = BN_;
    // Per-row A scale lines (per-token scales on the native path): 32 distinct
    // 16-byte lines per 128-K half instead of 8 identical ones.
    static constexpr bool ROWA = ROWA_;
    static constexpr bool PAIR = PAIR_;   // CTA pair (cta_group::2): 256-row tiles, B split by columns
    // Grouped (decode) tiles are 64 rows high: the A slots hold 64 rows, which
    // leaves room for a fifth operand stage (more weight bytes in flight).  The
    // M=128 MMA then also reads the 64 rows of shared memory after the slot;
    // those accumulator rows are never stored.
    static constexpr bool GROUPED = GROUPED_;
    static constexpr int TILE_M = PAIR ? 2 * BM : (GROUPED ? BM / 2 : BM);   // output rows per tile
    static constexpr int MMA_M = PAIR ? 2 * BM : BM;                // rows of every MMA instruction
    // Wide operand stages (CTA pairs) hold two 128-K halves ([half][rows][128
    // B], each a 128-byte-swizzled K-major slice) that arrive as one 3D TMA box
    // per operand: under load the TMA unit's per-request cost dominates, so
    // fewer, larger requests keep the loads ahead of the tensor cores.  One
    // scale-ring entry covers one operand stage, so the scale warp and the MMA
    // thread pay their barrier round trips once per 256 K.
    static constexpr bool WIDE = PAIR;
    static constexpr int HALVES = WIDE ? 2 : 1;
    static constexpr int STAGES = PAIR ? 3 : (GROUPED ? 5 : ((BN == 256) ? 4 : 6));
    static constexpr int A_HALF = (GROUPED ? BM / 2 : BM) * BK;     // this CTA's A rows, one 128-K half
    static constexpr int B_HALF = (PAIR ? BN / 2 : BN) * BK;        // this CTA's B rows, one 128-K half
    static constexpr int A_BYTES = HALVES * A_HALF;                 // per operand stage
    static constexpr int B_BYTES = HALVES * B_HALF;
    static constexpr int SFB_CHUNKS = (BN + 127) / 128;           // 128 B rows per tcgen05.cp
    static constexpr int SF_SET = 128;                              // 8 lines x 16 B, read 4 times by tcgen05.cp
    static constexpr int SF_SET_A = ROWA ? 512 : SF_SET;            // A's lines: 32 distinct or 8 identical
    static constexpr int SF_BYTES = SF_SET_A + SF_SET * SFB_CHUNKS; // scale lines per 128-K half
    static constexpr int SF_COLS = 4 * (1 + SFB_CHUNKS);            // tensor-memory columns per stage
    static constexpr int SF_STAGES = PAIR ? 9 : 8;                  // scale ring entries (runs ahead of the
                                                                    // operand ring)
    static constexpr int SF_ENTRY = HALVES * SF_BYTES;              // lines of one entry
    static constexpr int SF_ENTRY_COLS = HALVES * SF_COLS;
    static constexpr int SF_COL0 = (2 * BN + SF_STAGES * SF_ENTRY_COLS <= 512) ? 2 * BN : BN;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_COLS = BN / 2;                         // columns per epilogue warp
    // output staging for TMA stores: per column half, BM rows x 32 bf16 columns
    static constexpr int STG_COLS = 32;
    static constexpr int STG_BYTES = 2 * BM * STG_COLS * 2;
    static constexpr int NBB = BN / 32;                             // 32-column blocks per tile
    static constexpr int SC_FLOATS = 16 + 4 * NBB;                  // staged fp32 scales per 128-K half
    static constexpr int SC_ENTRY = HALVES * SC_FLOATS;
    static_assert(SF_COL0 + SF_STAGES * SF_ENTRY_COLS <= 512 && SF_COL0 >= BN, "tensor memory budget");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
    static_assert(4 * NBB <= 32, "one scale lane per 32-column block");
};

struct GroupEntry {
    const uint8_t *A;
    const float *sA;
    const float *sB;
    __nv_bfloat16 *C;
};

struct Common {
    int M, N, K, KB, KS;     // KB = K/32, KS = stages per tile
    int mt, nt, num_tiles;   // plain problem tiling
    int mode;
    int G;
    const int32_t *Ms;       // grouped: device row counts
    uint32_t *status;
    long long wait_limit;
    int withhold_stage;
    unsigned long long *trace;   // optional event trace of CTA 0 (see trace_event)
};

// Event trace (profiling aid, off when the pointer is null): CTA 0 records the
// SM clock of pipeline events into trace[event * TRACE_SLOTS + index].  The
// MMA thread records per-tile events only: a test of the trace pointer between
// a stage's MMAs costs ~3 % of the prefill GEMM (events 3, 4, 13 and 14 are
// unused).
constexpr int TRACE_SLOTS = 1024;
enum : int {
    TR_PROD_ISSUE = 0,      // producer: slot free, issuing stage `it`
    TR_SCALE_FULL = 1,      // scale warp: stage `it` landed
    TR_SCALE_READY = 2,     // scale warp: stage `it` lines written, released
    TR_EPI_FULL = 5,        // epilogue warp 4: accumulator of tile `i` ready
    TR_EPI_RELEASED = 6,    // epilogue warp 4: accumulator of tile `i` released
    TR_EPI_STORED = 7,      // epilogue warp 4: tile `i` stored
    TR_VERDICT = 8,         // verdict warp: tile `i` published
    TR_MMA_TILE = 9,        // MMA lane 0: tile `i` accumulator free, starting
    TR_PROD_TMA = 10,       // producer: stage `it` TMA issued
    TR_SCALE_ISSUE = 11,    // scale warp: entry free, issuing the copies of step `it`
    TR_SCALE_BUILD = 12,    // scale warp: starting step `it`'s lines (before waiting for its copies)
    TR_PEER_FWD = 15,       // peer MMA warp: its scale lines of stage `it` forwarded
    TR_MMA_VOK = 16,        // MMA lane 0: verdict of tile `i` seen
    TR_MMA_T0 = 17,         // MMA lane 0: accumulator released by the local epilogue (tile `i`)
    TR_MMA_LOOP = 18,       // MMA lane 0: tile `i`'s K loop about to wait for its first scale entry
    TR_EVENTS = 24
};

// CTA 1 (the pair peer when CTAs are paired) records at event + TR_EVENTS.
__device__ __forceinline__ void trace_event(const Common &c, int ev, int idx) {
    if (c.trace != nullptr && blockIdx.x < 2 && idx >= 0 && idx < TRACE_SLOTS)
        c.trace[(ev + static_cast<int>(blockIdx.x) * TR_EVENTS) * TRACE_SLOTS + idx] =
            static_cast<unsigned long long>(clock64());
}

struct PlainArgs {
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmC;    // bf16 output {N, M}, box {32, 128}: epilogue TMA stores
    CUtensorMap tmA3;   // wide stages: {128 K bytes, rows, K/128 halves} views of A and B
    CUtensorMap tmB3;
    GroupEntry e;
    Common c;
    CUtensorMap tmR;    // residual kernels: bf16 residual, same shape and box as C
    const __nv_bfloat16 *R;
    CUtensorMap tmQ;    // quantized-output kernels: E4M3 codes {N, M} bytes, box {32, 128}
    uint8_t *Cq;        //   the codes [M][N] and the block scales [ceil(M/32)][N/32]
    float *sC;
};

struct GroupedArgs {
    CUtensorMap tmB[MAX_GROUPS];
    GroupEntry e[MAX_GROUPS];
    Common c;
};

// One group's record in device memory (the C ABI's fp8_group_desc layout).
struct GroupRecord {
    const uint8_t *A;
    const float *sA;
    const uint8_t *B;
    const float *sB;
    __nv_bfloat16 *C;
};

// Grouped problems whose records live in device memory: the group table may
// change between launches (or CUDA-graph replays) without the host.  The B
// tensor maps are built on the device from a template by
// bsfp8_grouped_prepare, which also checks each record.
struct GroupedDevArgs {
    const GroupRecord *table;   // [G] records
    const CUtensorMap *maps;    // [G] B tensor maps (written by the prepare kernel)
    const int32_t *valid;       // [G] 1: the record passed the checks; 0: the group is skipped
    Common c;
};

__device__ __forceinline__ GroupEntry group_entry(const GroupedArgs &a, int g) { return a.e[g]; }
__device__ __forceinline__ GroupEntry group_entry(const GroupedDevArgs &a, int g) {
    const GroupRecord r = a.table[g];
    return GroupEntry{r.A, r.sA, r.sB, r.C};
}
__device__ __forceinline__ const CUtensorMap *group_bmap(const GroupedArgs &a, int g) { return &a.tmB[g]; }
__device__ __forceinline__ const CUtensorMap *group_bmap(const GroupedDevArgs &a, int g) { return a.maps + g; }
__device__ __forceinline__ bool group_valid(const GroupedArgs &, int) { return true; }
__device__ __forceinline__ bool group_valid(const GroupedDevArgs &a, int g) { return a.valid[g] != 0; }
template <typename Args> struct DevTable { static constexpr bool value = false; };
template <> struct DevTable<GroupedDevArgs> { static constexpr bool value = true; };

template <int STAGES, int SF_STAGES>
struct Ctrl {
    uint64_t full[STAGES];        // producer -> MMA warp (TMA bytes; grouped: + A-row cp.async;
                                  // pairs: both CTAs' bytes, on the leader's copy)
    uint64_t empty[STAGES];       // MMA commit -> producer
    uint64_t scfull[SF_STAGES];   // scale cp.async landed -> scale warp
    uint64_t sfready[SF_STAGES];  // scale warp -> MMA warp (lines written)
    uint64_t sfempty[SF_STAGES];  // MMA commit -> scale warp (lines and scales consumed)
    uint64_t tfull[2];          // MMA commit -> epilogue (accumulator / partial b)
    uint64_t tempty[2];         // epilogue -> MMA
    uint64_t vfull[2];          // verdict -> MMA, scale and epilogue warps
    uint64_t vempty[2];
    uint64_t drain;
    uint64_t rfull[2];          // residual chunk of column half h landed in its staging buffer
    uint32_t tmem_base;
    int verdict[2];
    int first_bad;              // the CTA's first tile reads a non-power-of-two scale
    int abort;
    int num_tiles;
    int tile_start[MAX_GROUPS + 1];
    int mg[MAX_GROUPS];
};

struct Tile {
    int m0, n0, Mg, g;
};

template <int BN, bool PAIR = false, bool GROUPED = false, bool ROWA = false>
constexpr int smem_bytes() {
    using C = Cfg<BN, PAIR, GROUPED, ROWA>;
    return 1024 + C::STAGES * (C::A_BYTES + C::B_BYTES) + C::STG_BYTES +
           C::SF_STAGES * (C::SF_ENTRY + 4 * C::SC_ENTRY) +
           static_cast<int>(sizeof(Ctrl<C::STAGES, C::SF_STAGES>));
}

// ---------------------------------------------------------------------------
// Bounded wait.  The waiting threads are parked in hardware (try_wait with a
// suspend hint) rather than polling: many warps spinning on barriers would
// take the shared-memory issue path away from the producer and MMA warps.
// The abort flag and the clock budget are looked at between suspensions.
constexpr uint32_t kSuspendHintNs = 200000;   // 0.2 ms per suspension at most
template <typename CtrlT>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, CtrlT *ctl,
                                         const Common &c) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
        if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
        if (clock64() - t0 > c.wait_limit) {
            *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
            atomicOr(c.status, STATUS_TIMEOUT);
            return false;
        }
    }
}

// Latency-critical wait of the single MMA-issuing thread: polls without
// suspending (a woken thread resumes a few hundred cycles late) and looks at
// the clock / abort flag every 256 polls.
template <typename CtrlT>
__device__ __forceinline__ bool wait_spin(uint64_t *bar, uint32_t parity, CtrlT *ctl,
                                          const Common &c) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((n & 255u) == 0u) {
            if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
            if (clock64() - t0 > c.wait_limit) {
                *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
                atomicOr(c.status, STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

// Wait of the epilogue warps for a finished accumulator: polls with short
// sleeps.  A thread parked in try_wait can resume thousands of cycles after the
// phase completes, and the next tile's MMAs wait for these warps' release.
template <typename CtrlT>
__device__ __forceinline__ bool wait_poll(uint64_t *bar, uint32_t parity, CtrlT *ctl,
                                          const Common &c) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        __nanosleep(100);
        if (mbar_test_wait(bar, parity)) return true;
        if ((n & 63u) == 0u) {
            if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
            if (clock64() - t0 > c.wait_limit) {
                *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
                atomicOr(c.status, STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

// Wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ bool wait_bar_drain(uint64_t *bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

__device__ __forceinline__ bool is_pow2_scale(float v) {
    const uint32_t b = __float_as_uint(v);
    const uint32_t e = b >> 23;   // sign must be 0, so this is the exponent
    return (b & 0x007FFFFFu) == 0u && e != 0u && e < 255u;
}

__device__ __forceinline__ uint32_t ue8m0_of(float v) { return (__float_as_uint(v) >> 23) & 0xFFu; }


template <int BN, bool GROUPED, typename Args, int TILE_M = BM>
struct Sched {
    const Args &a;
    const Common c;          // a copy in registers: the kernel parameters sit behind
                             // generic loads once the argument block's address is taken
    const int *tile_start;
    const int *mg;

    __device__ __forceinline__ Tile tile(int t) const {
        Tile r;
        if constexpr (!GROUPED) {
            const int per_group = GROUP_M * c.nt;
            const int grp = t / per_group;
            const int first_m = grp * GROUP_M;
            const int gsz = min(c.mt - first_m, GROUP_M);
            const int in = t - grp * per_group;
            r.m0 = (first_m + in % gsz) * TILE_M;
            r.n0 = (in / gsz) * BN;
            r.Mg = c.M;
            r.g = 0;
        } else {
            int lo = 0, hi = c.G - 1;   // last g with tile_start[g] <= t
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
            }
            const int g = lo;
            const int Mg = mg[g];
            const int mtg = (Mg + TILE_M - 1) / TILE_M;
            const int local = t - tile_start[g];
            r.m0 = (local % mtg) * TILE_M;
            r.n0 = (local / mtg) * BN;
            r.Mg = Mg;
            r.g = g;
        }
        return r;
    }

    GroupEntry e0;           // plain problems: the one entry, in registers

    __device__ __forceinline__ GroupEntry entry(int g) const {
        if constexpr (!GROUPED) return e0;
        else return group_entry(a, g);
    }
};

// True when any scale the tile reads is not a positive normal power of two.
// The tile's scales are two contiguous ranges (sA rows mb0..mb1 and sB rows
// nb0..nb1, all K blocks); thread t of n scans elements t, t + n, ..., with
// 16 loads in flight per round (the first tile's scan is a cold DRAM read).
template <int BN, int TILE_M>
__device__ __forceinline__ bool tile_has_bad_scale(const Tile &tt, const GroupEntry &e, const Common &c,
                                                   int t, int n) {
    const int MB = (tt.Mg + 31) / 32;
    const int mb0 = tt.m0 / 32, mb1 = min(mb0 + TILE_M / 32, MB);
    const int nb0 = tt.n0 / 32, nb1 = min(nb0 + BN / 32, c.N / 32);
    const float *pa = e.sA + static_cast<int64_t>(mb0) * c.KB;
    const int na = (mb1 - mb0) * c.KB;
    const float *pb = e.sB + static_cast<int64_t>(nb0) * c.KB;
    const int total = na + (nb1 - nb0) * c.KB;
    constexpr int U = 16;
    bool bad = false;
    for (int x0 = t; x0 < total; x0 += n * U) {
        float v[U];
#pragma unroll
        for (int w = 0; w < U; ++w) {
            const int x = x0 + w * n;
            v[w] = x < na ? __ldg(pa + x) : (x < total ? __ldg(pb + (x - na)) : 1.0f);
        }
#pragma unroll
        for (int w = 0; w < U; ++w) bad |= !is_pow2_scale(v[w]);
    }
    return bad;
}

// 32 consecutive bf16 outputs (64 bytes, 16-byte aligned) from fp32 bits / values.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const uint32_t *r) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 2 * x]),
                                                      __uint_as_float(r[8 * w + 2 * x + 1]));
            o[x] = *reinterpret_cast<uint32_t *>(&pr);
        }
        d[w] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// 32 fp32 bit patterns -> 32 bf16 (round to nearest even) into 64 bytes of shared memory.
__device__ __forceinline__ void pack_bf16x32(uint4 *dst, const uint32_t *r) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 2 * x]),
                                                      __uint_as_float(r[8 * w + 2 * x + 1]));
            o[x] = *reinterpret_cast<uint32_t *>(&pr);
        }
        dst[w] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// r[j] (fp32 bits) += the 32 bf16 values in 64 bytes of shared memory.
__device__ __forceinline__ void add_bf16x32(uint32_t *r, const uint4 *src) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint4 u = src[w];
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r[8 * w + 2 * k] = __float_as_uint(__uint_as_float(r[8 * w + 2 * k]) + __uint_as_float(wv[k] << 16));
            r[8 * w + 2 * k + 1] =
                __float_as_uint(__uint_as_float(r[8 * w + 2 * k + 1]) + __uint_as_float(wv[k] & 0xFFFF0000u));
        }
    }
}

__device__ __forceinline__ void store_bf16x32f(__nv_bfloat16 *dst, const float *v) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * w + 2 * x], v[8 * w + 2 * x + 1]);
            o[x] = *reinterpret_cast<uint32_t *>(&pr);
        }
        d[w] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// 32 fp32 values (bits or floats) -> 16 words of bf16 pairs (nearest even), or
// zeros for a row that does not exist.
__device__ __forceinline__ void bf16_words32(uint32_t (&o)[16], const uint32_t *r, bool keep) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        o[j] = keep ? *reinterpret_cast<uint32_t *>(&pr) : 0u;
    }
}
__device__ __forceinline__ void bf16_words32f(uint32_t (&o)[16], const float *v, bool keep) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        o[j] = keep ? *reinterpret_cast<uint32_t *>(&pr) : 0u;
    }
}

// One-CTA / CTA-pair forms of the tensor-core issue steps.
template <bool PAIR>
__device__ __forceinline__ void cp_lines(uint32_t taddr, uint64_t sdesc) {
    if constexpr (PAIR) tmem_cp_32x128b_warpx4_pair(taddr, sdesc);
    else tmem_cp_32x128b_warpx4(taddr, sdesc);
}
template <bool PAIR>
__device__ __forceinline__ void mma_block(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t acc) {
    if constexpr (PAIR) mma_mxf8_pair(d, ad, bd, idesc, sfa, sfb, acc);
    else mma_mxf8(d, ad, bd, idesc, sfa, sfb, acc);
}
// commit of all earlier tensor-core work to a barrier (both CTAs' copies for a pair)
template <bool PAIR>
__device__ __forceinline__ void commit_to(uint64_t *bar) {
    if constexpr (PAIR) mma_commit_pair(bar, 0x3);
    else mma_commit(bar);
}

// The scale copies and block-scaled MMAs of one operand stage (nk of its K
// blocks present; acc0: the stage's first MMA accumulates).  FULL stages are
// issued as one straight line: the tensor pipe holds about one MMA, so a
// branch between two MMAs delays the second one's issue past the first one's
// end (a full stage measured ~5 % faster on the prefill GEMM without them).
// Wide full stages also test the next stage's two barriers (nb0/np0,
// nb1/np1) inside the asm block of their last two MMAs and return the result
// (3.5-4.8 % on the prefill GEMM against a test after the commits); other
// stages return 0 and the caller tests after them.
template <typename C, bool FULL>
__device__ __forceinline__ uint32_t issue_native_stage(uint32_t tmem, uint32_t sfa, uint32_t sf_s, uint64_t ad,
                                                       uint64_t bd, int nk, uint32_t acc0, uint64_t *nb0,
                                                       uint32_t np0, uint64_t *nb1, uint32_t np1) {
    constexpr bool TAIL_TEST = FULL && C::HALVES == 2;
#pragma unroll
    for (int hh = 0; hh < C::HALVES; ++hh) {
        if (FULL || hh * KB_PER_STAGE < nk) {
            cp_lines<C::PAIR>(sfa + hh * C::SF_COLS, C::ROWA ? sdesc_sf_lines32(sf_s + hh * C::SF_BYTES)
                                                             : sdesc_sf_lines(sf_s + hh * C::SF_BYTES));
#pragma unroll
            for (int q = 0; q < C::SFB_CHUNKS; ++q)
                cp_lines<C::PAIR>(sfa + hh * C::SF_COLS + 4 + 4 * q,
                                  sdesc_sf_lines(sf_s + hh * C::SF_BYTES + C::SF_SET_A + C::SF_SET * q));
        }
    }
#pragma unroll
    for (int hh = 0; hh < C::HALVES; ++hh) {
#pragma unroll
        for (int j = 0; j < KB_PER_STAGE; ++j) {
            if (TAIL_TEST && hh == 1 && j >= KB_PER_STAGE - 2) continue;   // issued with the test below
            if (FULL || hh * KB_PER_STAGE + j < nk)
                mma_block<C::PAIR>(tmem, ad + static_cast<uint64_t>((hh * C::A_HALF >> 4) + 2 * j),
                                   bd + static_cast<uint64_t>((hh * C::B_HALF >> 4) + 2 * j),
                                   idesc_mxf8f6f4(C::MMA_M, C::BN, j, j), sfa + hh * C::SF_COLS,
                                   sfa + hh * C::SF_COLS + 4, (hh | j) != 0 ? 1u : acc0);
        }
    }
    if constexpr (TAIL_TEST) {
        constexpr int j0 = KB_PER_STAGE - 2, j1 = KB_PER_STAGE - 1;
        return mma_mxf8_x2_test<C::PAIR>(
            tmem, ad + static_cast<uint64_t>((C::A_HALF >> 4) + 2 * j0), bd + static_cast<uint64_t>((C::B_HALF >> 4) + 2 * j0),
            idesc_mxf8f6f4(C::MMA_M, C::BN, j0, j0), ad + static_cast<uint64_t>((C::A_HALF >> 4) + 2 * j1),
            bd + static_cast<uint64_t>((C::B_HALF >> 4) + 2 * j1), idesc_mxf8f6f4(C::MMA_M, C::BN, j1, j1),
            sfa + C::SF_COLS, sfa + C::SF_COLS + 4, nb0, np0, nb1, np1);
    } else {
        return 0u;
    }
}

// ---------------------------------------------------------------------------
// SK: scale layout; RES: a bf16 residual is added before the bf16 rounding;
// QOUT: the bf16 output is quantized to E4M3 codes with one scale per 32 x 32
// block (the block quantizer's arithmetic) instead of being stored.
template <int BN, bool GROUPED, bool PAIR, typename Args, int SK = SCALE_BLOCK32, bool RES = false,
          bool QOUT = false>
__device__ __forceinline__ void gemm_body(const Args &args, uint8_t *smem_raw) {
    static_assert(!QOUT || (PAIR && !RES && SK == SCALE_BLOCK32), "quantized output: block-scaled pair kernel");
    // per-token scales run the native path on CTA pairs (per-row scale lines)
    // and the promotion path on single CTAs
    using C = Cfg<BN, PAIR, GROUPED, PAIR && (SK == SCALE_TOKEN || SK == SCALE_TOKEN_E8)>;
    static_assert(SK != SCALE_TOKEN_E8 || PAIR, "UE8M0 per-token scales: CTA pairs");
    static_assert(!(PAIR && GROUPED), "CTA pairs are used for single problems only");
    constexpr int S = C::STAGES;
    constexpr int NBB = C::NBB;
    constexpr uint32_t FULL = 0xFFFFFFFFu;
    const Common c = args.c;   // register copy (see Sched)

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::A_BYTES;
    __nv_bfloat16 *sm_stg = reinterpret_cast<__nv_bfloat16 *>(sm_b + S * C::B_BYTES);   // [2][BM][STG_COLS]
    uint8_t *sm_sf = sm_b + S * C::B_BYTES + C::STG_BYTES;                   // [FS][HALVES][SF_BYTES]
    constexpr int FS = C::SF_STAGES;
    float *sm_sc = reinterpret_cast<float *>(sm_sf + FS * C::SF_ENTRY);      // [FS][HALVES][SC_FLOATS]
    using CtrlT = Ctrl<S, FS>;
    CtrlT *ctl = reinterpret_cast<CtrlT *>(sm_sc + FS * C::SC_ENTRY);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pairs: rank 0 (the leader) issues the pair's MMAs; each CTA owns
    // rows [rank*128, rank*128 + 128) of the tile and half of B's columns.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0u;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int grid_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int row_off = static_cast<int>(rank) * BM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // full: lane 0's expect_tx arrival (+ one A-row cp.async arrival per
            // producer lane for grouped problems); scfull: one scale cp.async
            // arrival per producer lane
            mbar_init(&ctl->full[s], GROUPED ? 1 + 32 : 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int f = 0; f < FS; ++f) {
            mbar_init(&ctl->scfull[f], 32);   // one cp.async arrival per scale-warp lane
            // the leader also waits for the peer's lines; per-row A lines are
            // written by warp 2 besides the scale warp
            mbar_init(&ctl->sfready[f], ((PAIR && leader) ? 2 : 1) + (C::ROWA ? 1 : 0));
            mbar_init(&ctl->sfempty[f], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], (PAIR && leader) ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
            mbar_init(&ctl->vfull[b], 1);
            mbar_init(&ctl->vempty[b], 2 + NUM_EPI_WARPS);   // MMA + scale warp + epilogue
        }
        mbar_init(&ctl->drain, 1);
        mbar_init(&ctl->rfull[0], 1);
        mbar_init(&ctl->rfull[1], 1);
        ctl->abort = 0;
        ctl->first_bad = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&ctl->tmem_base, C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ctl->tmem_base, C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    if (warp == 2) {
        if constexpr (GROUPED) {
            // tile table: group g owns tiles [tile_start[g], tile_start[g+1])
            if (lane == 0) {
                int acc = 0;
                for (int g = 0; g < c.G; ++g) {
                    int m = group_valid(args, g) ? c.Ms[g] : 0;   // a rejected record: no rows
                    m = m < 0 ? 0 : m;
                    ctl->mg[g] = m;
                    ctl->tile_start[g] = acc;
                    acc += ((m + C::TILE_M - 1) / C::TILE_M) * c.nt;
                }
                ctl->tile_start[c.G] = acc;
                ctl->num_tiles = acc;
            }
        } else {
            if (lane == 0) ctl->num_tiles = c.num_tiles;
        }
    }
    if (warp == 0) {
        if constexpr (!GROUPED) {
            if (lane == 0) {
                tma_prefetch_desc(&args.tmA);
                tma_prefetch_desc(&args.tmB);
                if constexpr (C::WIDE) {
                    tma_prefetch_desc(&args.tmA3);
                    tma_prefetch_desc(&args.tmB3);
                }
            }
        } else {
            if constexpr (!DevTable<Args>::value)
                for (int g = lane; g < c.G; g += 32) tma_prefetch_desc(group_bmap(args, g));
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before any remote arrive
    tc_fence_after();

    const uint32_t tmem = ctl->tmem_base;
    const int num_tiles = ctl->num_tiles;
    // Grouped launches use only as many CTAs as give each the same number of
    // tiles (the tile count is known here, from the device row counts): a last
    // round with fewer CTAs than the others measured slower (16 groups of
    // 4096 x 7168 weights, 256 tiles: 128 CTAs with two each take 90 us, 152
    // CTAs of which 104 take a second tile 93 us).
    int nunits = grid_units;
    if constexpr (GROUPED) {
        const int rounds = (num_tiles + grid_units - 1) / grid_units;
        nunits = rounds > 0 ? (num_tiles + rounds - 1) / rounds : grid_units;
    }
    const int my_tiles = (unit < num_tiles && unit < nunits) ? (num_tiles - unit + nunits - 1) / nunits : 0;
    GroupEntry e0{};
    if constexpr (!GROUPED) e0 = args.e;
    const Sched<BN, GROUPED, Args, C::TILE_M> sch{args, c, ctl->tile_start, ctl->mg, e0};
    constexpr uint16_t PAIR_MASK = 0x3;

    // The first tile's path verdict gates its MMAs and its scale lines.  Ten
    // warps compute it together (one or two rounds of loads instead of the
    // verdict warp's many) while the producer warp starts loading operands and
    // the scale warp its first scale copies.
    if (warp != 0 && warp != 3) {
        constexpr int SCANNERS = NUM_THREADS - 64;
        bool bad = false;
        if (my_tiles > 0 && c.mode != PATH_PROMOTE && SK == SCALE_BLOCK32) {
            const Tile tt = sch.tile(unit);
            const int t = static_cast<int>(threadIdx.x) - (warp < 3 ? 32 : 64);
            bad = tile_has_bad_scale<BN, C::TILE_M>(tt, sch.entry(tt.g), c, t, SCANNERS);
        }
        if (__any_sync(FULL, bad) && lane == 0) atomicOr(&ctl->first_bad, 1);
        named_bar_sync(1, SCANNERS);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Per stage only: wait for the slot, register the bytes, issue the
        // TMA; tile coordinates are decoded once per tile (a single warp runs
        // dependent integer chains slowly, so the per-stage path stays short).
        int it = 0, s = 0;   // it: operand stages issued (each HALVES x 128 K)
        uint32_t ph = 0;
        int withheld = -1;   // slot never armed (test hook), excluded from the drain
        bool ok = true;
        const int KW = (c.KS + C::HALVES - 1) / C::HALVES;   // operand stages per tile
        for (int i = 0; i < my_tiles && ok; ++i) {
            const Tile tt = sch.tile(unit + i * nunits);
            const GroupEntry e = sch.entry(tt.g);
            const CUtensorMap *tmb;
            if constexpr (GROUPED) tmb = group_bmap(args, tt.g);
            else tmb = &args.tmB;
            // a map written on the device: its writes are acquired before use
            if constexpr (DevTable<Args>::value) if (lane == 0) tensormap_acquire(tmb);
            const int a_rows = min(C::TILE_M, tt.Mg - tt.m0);   // grouped: A rows loaded by cp.async
            const uint8_t *a_base = e.A + static_cast<int64_t>(tt.m0) * c.K;
            for (int ks = 0, k0 = 0; ks < KW; ++ks, k0 += C::HALVES * BK) {
                ok = __all_sync(FULL, wait_bar(&ctl->empty[s], ph ^ 1u, ctl, c));
                if (!ok) break;
                if ((c.withhold_stage == it) && blockIdx.x < (PAIR ? 2u : 1u)) {
                    withheld = s;
                } else {
                    if (lane == 0) {
                        trace_event(c, TR_PROD_ISSUE, it);
                        if constexpr (PAIR) {
                            // both CTAs' loads complete on the leader's barrier
                            // (cta_group::2), which the leader arms for the pair's bytes
                            const int ar = tt.m0 + row_off, br = tt.n0 + static_cast<int>(rank) * (BN / 2);
                            const uint32_t bar_l = mapa_shared(&ctl->full[s], 0);   // the leader's barrier
                            if (k0 + 2 * BK <= c.K) {
                                // both halves inside K: one box per operand
                                if (leader) mbar_arrive_expect_tx(&ctl->full[s], 2 * (C::A_BYTES + C::B_BYTES));
                                tma_load_3d_pair(&args.tmA3, bar_l, sm_a + s * C::A_BYTES, 0, ar, k0 / BK);
                                tma_load_3d_pair(&args.tmB3, bar_l, sm_b + s * C::B_BYTES, 0, br, k0 / BK);
                            } else {
                                // the tile's last stage: the halves that start before K,
                                // from the 2D maps, which zero-fill K past the end
                                const int nh = k0 + BK < c.K ? 2 : 1;
                                if (leader) mbar_arrive_expect_tx(&ctl->full[s], 2 * nh * (C::A_HALF + C::B_HALF));
                                for (int hh = 0; hh < nh; ++hh) {
                                    tma_load_2d_pair(&args.tmA, bar_l, sm_a + s * C::A_BYTES + hh * C::A_HALF,
                                                     k0 + hh * BK, ar);
                                    tma_load_2d_pair(tmb, bar_l, sm_b + s * C::B_BYTES + hh * C::B_HALF,
                                                     k0 + hh * BK, br);
                                }
                            }
                        } else {
                            if constexpr (!GROUPED) {
                                mbar_arrive_expect_tx(&ctl->full[s], C::A_BYTES + C::B_BYTES);
                                tma_load_2d(&args.tmA, &ctl->full[s], sm_a + s * C::A_BYTES, k0, tt.m0);
                            } else {
                                mbar_arrive_expect_tx(&ctl->full[s], C::B_BYTES);
                            }
                            tma_load_2d(tmb, &ctl->full[s], sm_b + s * C::B_BYTES, k0, tt.n0);
                        }
                        trace_event(c, TR_PROD_TMA, it);
                    }
                    if constexpr (GROUPED) {
                        // A rows of this group: 16-byte cp.async into the 128-byte
                        // swizzled layout; chunks past K are zero-filled, rows past
                        // M_g are not loaded (they only feed output rows that are
                        // never stored).
                        const uint32_t dst0 = smem_u32(sm_a + s * C::A_BYTES);
                        for (int idx = lane; idx < a_rows * 8; idx += 32) {
                            const int r = idx >> 3, ch = idx & 7;
                            const int kk = k0 + ch * 16;
                            const bool in = kk < c.K;
                            cp_async_16(dst0 + r * 128 + ((ch ^ (r & 7)) << 4),
                                        a_base + static_cast<int64_t>(r) * c.K + (in ? kk : 0), in ? 16u : 0u);
                        }
                        cp_async_mbar_arrive_noinc(&ctl->full[s]);
                    }
                }
                ++it;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
        // drain: every armed stage's last phase must complete before the CTA exits
        // (a pair's loads all complete on the leader's barriers)
        if (lane == 0 && (!PAIR || leader)) {
            for (int d = max(0, it - S); d < it; ++d) {
                const int sd = d % S;
                if (sd == withheld) continue;
                wait_bar_drain(&ctl->full[sd], static_cast<uint32_t>(d / S) & 1u, c.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA warp
        // One thread runs the role: the warp's other lanes wait at the end, so
        // no tile boundary pays a warp-wide reconvergence.
        if (lane == 0) {
            int ot = 0;                       // operand stages consumed (the producer's sequence)
            const int KW = (c.KS + C::HALVES - 1) / C::HALVES;
            uint32_t uses0 = 0, uses1 = 0;    // completed uses of tensor-memory buffers 0 / 1
            uint32_t pk = 0;                  // promotion partials issued (buffer = pk & 1)
            // Promotion tiles: the epilogue reads each K block's scales from the
            // scale ring, so an entry is released (sfempty) only once the epilogue
            // has read every partial of its stage.  The MMA thread learns that from
            // its own tempty waits (the wait for partial p passes once partial p-2
            // has been read); entries wait here, oldest first, with the index of
            // their last partial.
            int pend_f0 = -1, pend_l0 = 0, pend_f1 = -1, pend_l1 = 0;
            // A pair's peer: in promotion tiles its epilogue releases a partial on
            // its own barrier only, and this thread, which waits there anyway,
            // forwards the release to the leader as one arrival counting for the
            // peer's eight warps (bit b: buffer b's last use still to forward).
            uint32_t fwd = 0;
            auto forward_release = [&](uint32_t b) {
                if (PAIR && !leader && ((fwd >> b) & 1u)) {
                    mbar_signal_cluster_count(mapa_shared(&ctl->tempty[b], 0), NUM_EPI_WARPS);
                    fwd &= ~(1u << b);
                }
            };
            auto release_read = [&](int upto) {   // partials <= upto have been read
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (pend_f0 >= 0 && pend_l0 <= upto) {
                        mbar_arrive(&ctl->sfempty[pend_f0]);
                        pend_f0 = pend_f1;
                        pend_l0 = pend_l1;
                        pend_f1 = -1;
                    }
                }
            };
            bool ok = true;
            bool issued = false;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int v = i & 1;
                ok = wait_spin(&ctl->vfull[v], static_cast<uint32_t>(i >> 1) & 1u, ctl, c);
                if (!ok) break;
                const bool promote = ctl->verdict[v] != 0;
                if (!promote && pend_f0 >= 0) {
                    // a promotion tile's last scale entries: both buffers drained
                    // means every partial has been read
                    ok = wait_bar(&ctl->tempty[0], (uses0 & 1u) ^ 1u, ctl, c) &&
                         wait_bar(&ctl->tempty[1], (uses1 & 1u) ^ 1u, ctl, c);
                    if (!ok) break;
                    forward_release(0u);
                    forward_release(1u);
                    release_read(static_cast<int>(pk));
                }
                if (!promote) {
                    if (leader) {
                        trace_event(c, TR_MMA_VOK, i);
                        // the accumulator (buffer 0) and, since the scale columns
                        // share its range, buffer 1 must both be drained
                        ok = wait_spin(&ctl->tempty[0], (uses0 & 1u) ^ 1u, ctl, c);
                        trace_event(c, TR_MMA_T0, i);
                        ok = ok && wait_spin(&ctl->tempty[1], (uses1 & 1u) ^ 1u, ctl, c);
                        trace_event(c, TR_MMA_TILE, i);
                        tc_fence_after();
                        const uint32_t sfa_base = tmem + C::SF_COL0;
                        // one pass per operand stage: the MMA pipe holds only about one
                        // instruction, so the thread keeps the work between MMAs short
                        // (counters instead of divisions; all scale copies of the stage
                        // first, then its MMAs back to back; no trace events here)
                        int s = ot % S, f = ot % FS;
                        uint32_t ph = static_cast<uint32_t>(ot / S) & 1u, phf = static_cast<uint32_t>(ot / FS) & 1u;
                        trace_event(c, TR_MMA_LOOP, i);
                        // One operand stage: its barriers (unless the previous stage found
                        // them complete), scale copies and MMAs, commits; the next stage's
                        // barriers are tested without blocking (one test of both, with the
                        // last two MMAs on wide stages, else after the commits).  Each
                        // branch of this single thread costs tens of cycles in which the
                        // pipe may run dry.
                        bool next_ready = false;
                        auto stage = [&](auto full, int w) -> bool {
                            if (!next_ready &&
                                !(wait_spin(&ctl->sfready[f], phf, ctl, c) && wait_spin(&ctl->full[s], ph, ctl, c)))
                                return false;
                            if constexpr (GROUPED) fence_proxy_async_smem();   // A rows written by cp.async
                            tc_fence_after();
                            const uint32_t sfa = sfa_base + f * C::SF_ENTRY_COLS;
                            const uint32_t sf_s = smem_u32(sm_sf + f * C::SF_ENTRY);
                            const uint64_t ad = sdesc_k_sw128(smem_u32(sm_a + s * C::A_BYTES));
                            const uint64_t bd = sdesc_k_sw128(smem_u32(sm_b + s * C::B_BYTES));
                            const int nk = decltype(full)::value ? C::HALVES * KB_PER_STAGE
                                                                 : min(C::HALVES * KB_PER_STAGE, c.KB - w * C::HALVES * KB_PER_STAGE);
                            const int s2 = s + 1 == S ? 0 : s + 1, f2 = f + 1 == FS ? 0 : f + 1;
                            const uint32_t ph2 = ph ^ (s2 == 0 ? 1u : 0u), phf2 = phf ^ (f2 == 0 ? 1u : 0u);
                            uint32_t t = issue_native_stage<C, decltype(full)::value>(
                                tmem, sfa, sf_s, ad, bd, nk, w != 0 ? 1u : 0u, &ctl->sfready[f2], phf2, &ctl->full[s2], ph2);
                            commit_to<PAIR>(&ctl->empty[s]);
                            commit_to<PAIR>(&ctl->sfempty[f]);
                            s = s2;
                            f = f2;
                            ph = ph2;
                            phf = phf2;
                            if (!(decltype(full)::value && C::HALVES == 2)) t = mbar_test_wait2(&ctl->sfready[f], phf, &ctl->full[s], ph);
                            next_ready = (t != 0u) & (w + 1 < KW);
                            return true;
                        };
                        // Full stages first, as straight lines of copies and MMAs; a
                        // partial last stage (K not a multiple of 256) after them.  Per-token
                        // lines keep the guarded body for every stage: their stages wait
                        // for warp 2's scale loads, and the straight line measured 2-3 %
                        // slower there.
                        const int kw_full = C::ROWA ? 0 : c.KB / (C::HALVES * KB_PER_STAGE);
                        int w = 0;
                        for (; w < kw_full && ok; ++w) ok = stage(std::true_type{}, w);
                        for (; w < KW && ok; ++w) ok = stage(std::false_type{}, w);
                        issued = issued || KW > 0;
                        if (ok) commit_to<PAIR>(&ctl->tfull[0]);
                    }
                    if (PAIR && !leader) {
                        // forward each stage's scale lines to the leader's MMA thread
                        for (int w = 0; w < KW && ok; ++w) {
                            const int os = ot + w;
                            const int f = os % FS;
                            ok = wait_spin(&ctl->sfready[f], static_cast<uint32_t>(os / FS) & 1u, ctl, c);
                            if (ok) mbar_signal_cluster(mapa_shared(&ctl->sfready[f], 0));
                            trace_event(c, TR_PEER_FWD, os);
                        }
                    }
                    if (!ok) break;
                    ot += KW;
                    ++uses0;
                } else {
                    if (pk & 1u) ++pk;   // promotion tiles start on buffer 0 (see the header)
                    int s = ot % S, f = ot % FS;
                    uint32_t ph = static_cast<uint32_t>(ot / S) & 1u, phf = static_cast<uint32_t>(ot / FS) & 1u;
                    const int kw_full = c.KB / (C::HALVES * KB_PER_STAGE);
                    for (int w = 0; w < KW && ok; ++w) {
                        ok = (PAIR && !leader ? true : wait_bar(&ctl->full[s], ph, ctl, c)) &&
                             wait_bar(&ctl->sfready[f], phf, ctl, c);
                        if (!ok) break;
                        if (PAIR && !leader) mbar_signal_cluster(mapa_shared(&ctl->sfready[f], 0));
                        if constexpr (GROUPED) fence_proxy_async_smem();   // A rows written by cp.async
                        const uint64_t ad = sdesc_k_sw128(smem_u32(sm_a + s * C::A_BYTES));
                        const uint64_t bd = sdesc_k_sw128(smem_u32(sm_b + s * C::B_BYTES));
                        // partial j of the stage (K block j % 4 of half j / 4) into buffer b,
                        // once the epilogue has read that buffer's previous partial
                        auto partial = [&](int j, uint32_t b) -> bool {
                            if (!wait_bar(&ctl->tempty[b], ((b ? uses1 : uses0) & 1u) ^ 1u, ctl, c)) return false;
                            forward_release(b);
                            release_read(static_cast<int>(pk) - 2);
                            if (leader) {
                                const int hh = j / KB_PER_STAGE, jj = j % KB_PER_STAGE;
                                const uint64_t a_j = ad + static_cast<uint64_t>((hh * C::A_HALF >> 4) + 2 * jj);
                                const uint64_t b_j = bd + static_cast<uint64_t>((hh * C::B_HALF >> 4) + 2 * jj);
                                tc_fence_after();
                                if constexpr (PAIR) {
                                    mma_f8_pair(tmem + b * BN, a_j, b_j, idesc_f8f6f4(C::MMA_M, BN), 0u);
                                    mma_commit_pair(&ctl->tfull[b], PAIR_MASK);
                                } else {
                                    mma_f8(tmem + b * BN, a_j, b_j, idesc_f8f6f4(BM, BN), 0u);
                                    mma_commit(&ctl->tfull[b]);
                                }
                            }
                            issued = true;
                            if (b) ++uses1; else ++uses0;
                            fwd |= 1u << b;
                            ++pk;
                            return true;
                        };
                        if (w < kw_full) {
                            // a full stage: an even number of partials from an even pk, so
                            // partial j uses buffer j & 1 (known when the loop is unrolled)
#pragma unroll
                            for (int j = 0; j < C::HALVES * KB_PER_STAGE; ++j)
                                if (ok) ok = partial(j, static_cast<uint32_t>(j & 1));
                        } else {
                            const int nk = c.KB - w * C::HALVES * KB_PER_STAGE;
                            for (int j = 0; j < nk && ok; ++j) ok = partial(j, pk & 1u);
                        }
                        if (!ok) break;
                        if (leader) commit_to<PAIR>(&ctl->empty[s]);
                        // the stage's scale entry, released once its partials are read
                        if (pend_f0 < 0) { pend_f0 = f; pend_l0 = static_cast<int>(pk) - 1; }
                        else { pend_f1 = f; pend_l1 = static_cast<int>(pk) - 1; }
                        s = s + 1 == S ? 0 : s + 1;
                        ph ^= s == 0 ? 1u : 0u;
                        f = f + 1 == FS ? 0 : f + 1;
                        phf ^= f == 0 ? 1u : 0u;
                    }
                    if (!ok) break;
                    ot += KW;
                }
                mbar_arrive(&ctl->vempty[v]);
            }
            // all issued tensor-core work must finish before tensor memory is freed
            if (issued && leader) {
                if constexpr (PAIR) mma_commit_pair(&ctl->drain, 0x1);
                else mma_commit(&ctl->drain);
                wait_bar_drain(&ctl->drain, 0u, c.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        if constexpr (C::ROWA && SK == SCALE_TOKEN_E8) {
            // ------------------------------------ per-row A scale lines, UE8M0 bytes
            // As below, but sA holds the UE8M0 bytes themselves: lane l loads the
            // 8 bytes (one per 32-K block of the 256-K entry) of rows l, 32+l, 64+l
            // and 96+l, and word w of half h's line is bytes 4h..4h+3 of row 32w+l:
            // no conversion, and a quarter of the fp32 path's load bytes.  A byte
            // 0xFF (not a number in UE8M0) sets the status word's scale bit.
            constexpr int H = C::HALVES;
            static_assert(H == 2, "UE8M0 lines: 256-K entries");
            const int KW = (c.KS + H - 1) / H;
            const int total = my_tiles * KW;
            int il = -1, kl = KW;
            bool vec = false;   // every row starts on 8 bytes and holds whole entries
            const uint8_t *lp[4] = {nullptr, nullptr, nullptr, nullptr};
            auto load = [&](uint2 (&dst)[4]) {
                if (++kl >= KW) {
                    kl = 0;
                    ++il;
                    const Tile tt = sch.tile(unit + il * nunits);
                    const uint8_t *sa = reinterpret_cast<const uint8_t *>(sch.entry(tt.g).sA);
                    vec = (c.KB & 7) == 0 && (reinterpret_cast<uintptr_t>(sa) & 7u) == 0;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int row = tt.m0 + row_off + 32 * w + lane;
                        lp[w] = row < tt.Mg ? sa + static_cast<int64_t>(row) * c.KB : nullptr;
                    }
                }
                const int kb0 = kl * 8;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    if (vec) {
                        dst[w] = lp[w] != nullptr ? __ldg(reinterpret_cast<const uint2 *>(lp[w] + kb0))
                                                  : make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
                    } else {
                        uint32_t b[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            b[j] = (lp[w] != nullptr && kb0 + j < c.KB) ? __ldg(lp[w] + kb0 + j) : 0x7Fu;
                        dst[w] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                            b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
                    }
                }
            };
            int ib = -1, kbs = KW, fb = 0;
            uint32_t phb = 0;
            auto build = [&](const uint2 (&src)[4]) -> bool {
                if (++kbs >= KW) {
                    kbs = 0;
                    ++ib;
                    const int v = ib & 1;
                    if (!__all_sync(FULL, wait_bar(&ctl->vempty[v], (static_cast<uint32_t>(ib >> 1) & 1u) ^ 1u, ctl, c)))
                        return false;
                    if (lane == 0) {
                        ctl->verdict[v] = 0;
                        mbar_arrive(&ctl->vfull[v]);
                        trace_event(c, TR_VERDICT, ib);
                    }
                    __syncwarp();
                }
                const int f = fb;
                if (!__all_sync(FULL, wait_bar(&ctl->sfempty[f], phb ^ 1u, ctl, c))) return false;
                if (++fb == FS) {
                    fb = 0;
                    phb ^= 1u;
                }
                uint8_t *line = sm_sf + f * C::SF_ENTRY + lane * 16;
                *reinterpret_cast<uint4 *>(line) = make_uint4(src[0].x, src[1].x, src[2].x, src[3].x);
                *reinterpret_cast<uint4 *>(line + C::SF_BYTES) = make_uint4(src[0].y, src[1].y, src[2].y, src[3].y);
                // a byte 0xFF: its complement has a zero byte
                bool bad = false;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t x0 = ~src[w].x, x1 = ~src[w].y;
                    bad |= (((x0 - 0x01010101u) & ~x0 & 0x80808080u) | ((x1 - 0x01010101u) & ~x1 & 0x80808080u)) != 0u;
                }
                if (__any_sync(FULL, bad) && lane == 0) atomicOr(c.status, STATUS_SCALE);
                fence_proxy_async_smem();   // the lines become visible to tcgen05.cp
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sfready[f]);
                __syncwarp();
                return true;
            };
            // four entries in flight (an eight-deep unrolled ring measured 1386
            // against 1810 TFLOP/s on the 4096^3 GEMM)
            uint2 r0[4], r1[4], r2[4], r3[4];
            if (total > 0) load(r0);
            if (total > 1) load(r1);
            if (total > 2) load(r2);
            for (int e = 0; e < total; e += 4) {
                if (e + 3 < total) load(r3);
                if (!build(r0) || e + 1 >= total) break;
                if (e + 4 < total) load(r0);
                if (!build(r1) || e + 2 >= total) break;
                if (e + 5 < total) load(r1);
                if (!build(r2) || e + 3 >= total) break;
                if (e + 6 < total) load(r2);
                if (!build(r3)) break;
            }
        } else if constexpr (C::ROWA) {
            // ----------------------------------------------- per-row A scale lines
            // Per-token A scales (one per row per 32-K block) on the native path.
            // For each scale-ring entry lane l writes line l of each 128-K half:
            // word w holds the UE8M0 scales of row 32w + l of this CTA's 128 rows,
            // byte j that of K block j of the half, so tcgen05.cp hands every row
            // its own scales.  The scales of entry e + 3 are loaded (plain loads
            // into registers, four entries in flight: an L2 load under the
            // operand traffic takes about as long as a stage) before entry e's
            // lines are written; a scale that is not a positive normal power of
            // two sets the status word's scale bit.
            // Every tile's verdict is the native path; it is published when the
            // lines reach the tile (the verdict of tile i waits only for tile i - 2).
            constexpr int H = C::HALVES;
            const int KW = (c.KS + H - 1) / H;
            const int total = my_tiles * KW;
            // load side: tile il, stage kl of the entry being loaded; this lane's
            // four rows of that tile (null outside M); vec: every row of sA
            // starts on 16 bytes (the API promises only 4), one load per row and half
            int il = -1, kl = KW;
            bool vec = false;
            const float *lp[4] = {nullptr, nullptr, nullptr, nullptr};
            auto load = [&](float (&dst)[H][16]) {
                if (++kl >= KW) {
                    kl = 0;
                    ++il;
                    const Tile tt = sch.tile(unit + il * nunits);
                    const float *sa = sch.entry(tt.g).sA;
                    vec = (c.KB & 3) == 0 && (reinterpret_cast<uintptr_t>(sa) & 15u) == 0;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int row = tt.m0 + row_off + 32 * w + lane;
                        lp[w] = row < tt.Mg ? sa + static_cast<int64_t>(row) * c.KB : nullptr;
                    }
                }
                // each row's next 128-byte line (the scales of the next four
                // entries) goes to L1 ahead of its loads; one line ahead per row
                // is 16 KB, what L1 holds beside this kernel's shared memory
                if ((kl & 3) == 0) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int nl = (kl >> 2) + 1;
                        if (lp[w] != nullptr && nl * 32 < c.KB)
                            asm volatile("prefetch.global.L1 [%0];" ::"l"(lp[w] + nl * 32));
                    }
                }
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const int kb0 = (kl * H + h) * KB_PER_STAGE;
                        if (vec) {
                            const float4 q = (lp[w] != nullptr && kb0 < c.KB)
                                                 ? __ldg(reinterpret_cast<const float4 *>(lp[w] + kb0))
                                                 : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
                            dst[h][4 * w + 0] = q.x;
                            dst[h][4 * w + 1] = q.y;
                            dst[h][4 * w + 2] = q.z;
                            dst[h][4 * w + 3] = q.w;
                        } else {
#pragma unroll
                            for (int j = 0; j < KB_PER_STAGE; ++j)
                                dst[h][4 * w + j] =
                                    (lp[w] != nullptr && kb0 + j < c.KB) ? __ldg(lp[w] + kb0 + j) : 1.0f;
                        }
                    }
                }
            };
            // build side: tile ib, stage kbs, ring slot fb (phase phb)
            int ib = -1, kbs = KW, fb = 0;
            uint32_t phb = 0;
            auto build = [&](const float (&src)[H][16]) -> bool {
                if (++kbs >= KW) {
                    kbs = 0;
                    ++ib;
                    const int v = ib & 1;
                    if (!__all_sync(FULL, wait_bar(&ctl->vempty[v], (static_cast<uint32_t>(ib >> 1) & 1u) ^ 1u, ctl, c)))
                        return false;
                    if (lane == 0) {
                        ctl->verdict[v] = 0;
                        mbar_arrive(&ctl->vfull[v]);
                        trace_event(c, TR_VERDICT, ib);
                    }
                    __syncwarp();
                }
                const int f = fb;
                if (!__all_sync(FULL, wait_bar(&ctl->sfempty[f], phb ^ 1u, ctl, c))) return false;
                if (++fb == FS) {
                    fb = 0;
                    phb ^= 1u;
                }
                // a positive normal power of two has sign and mantissa zero and
                // 1 <= exponent <= 254; its UE8M0 byte is its exponent field, so
                // a word of four is assembled by shifts alone
                uint32_t mant = 0u, lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    uint32_t wd[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t b0 = __float_as_uint(src[h][4 * w + 0]), b1 = __float_as_uint(src[h][4 * w + 1]);
                        const uint32_t b2 = __float_as_uint(src[h][4 * w + 2]), b3 = __float_as_uint(src[h][4 * w + 3]);
                        mant |= (b0 | b1 | b2 | b3) & 0x807FFFFFu;
                        lo = min(lo, min(min(b0, b1), min(b2, b3)));
                        hi = max(hi, max(max(b0, b1), max(b2, b3)));
                        wd[w] = (b0 >> 23) | (b1 >> 15) | (b2 >> 7) | (b3 << 1);
                    }
                    *reinterpret_cast<uint4 *>(sm_sf + f * C::SF_ENTRY + h * C::SF_BYTES + lane * 16) =
                        make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
                const bool bad = mant != 0u || lo < 0x00800000u || hi >= 0x7F800000u;
                if (__any_sync(FULL, bad) && lane == 0) atomicOr(c.status, STATUS_SCALE);
                fence_proxy_async_smem();   // the lines become visible to tcgen05.cp
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sfready[f]);
                __syncwarp();
                return true;
            };
            float r0[H][16], r1[H][16], r2[H][16], r3[H][16];
            if (total > 0) load(r0);
            if (total > 1) load(r1);
            if (total > 2) load(r2);
            for (int e = 0; e < total; e += 4) {
                if (e + 3 < total) load(r3);
                if (!build(r0) || e + 1 >= total) break;
                if (e + 4 < total) load(r0);
                if (!build(r1) || e + 2 >= total) break;
                if (e + 5 < total) load(r1);
                if (!build(r2) || e + 3 >= total) break;
                if (e + 6 < total) load(r2);
                if (!build(r3)) break;
            }
        } else {
            // -------------------------------------------------------- path verdict
            for (int i = 0; i < my_tiles; ++i) {
                const int v = i & 1;
                bool ok = wait_bar(&ctl->vempty[v], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u, ctl, c);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                int verdict = 1;
                if constexpr (SK == SCALE_ROWCOL) {
                    verdict = 0;   // unit block scales: the native path
                } else if constexpr (SK == SCALE_TOKEN) {
                    verdict = 1;   // per-row scales: the promotion path
                } else if (c.mode != PATH_PROMOTE) {
                    bool any_bad;
                    if (i == 0) {
                        any_bad = ctl->first_bad != 0;   // computed by warps 1..11 at the start
                    } else {
                        const Tile tt = sch.tile(unit + i * nunits);
                        any_bad = __any_sync(FULL, tile_has_bad_scale<BN, C::TILE_M>(tt, sch.entry(tt.g), c, lane, 32));
                    }
                    verdict = any_bad ? 1 : 0;
                    if (any_bad && c.mode == PATH_NATIVE && lane == 0) atomicOr(c.status, STATUS_SCALE);
                }
                if (lane == 0) {
                    ctl->verdict[v] = verdict;
                    mbar_arrive(&ctl->vfull[v]);
                    trace_event(c, TR_VERDICT, i);
                }
                __syncwarp();
            }
        }
    } else if (warp == 3) {
        // --------------------------------------------------------- scale warp
        // One ring entry per operand stage (HALVES x 128 K).  Loads the
        // entry's fp32 block scales with cp.async -- per half h, lane l < 16:
        // sA[m0/32 + l/4][kb0 + 4h + l%4]; lane l < 4*BN/32: sB[n0/32 + l/4][kb0
        // + 4h + l%4], stored K-block-major (sA at [j][row block], sB at 16 +
        // [j][column block]) -- L entries ahead of turning them into the UE8M0
        // lines that tcgen05.cp replicates into all lane quarters.  Absent blocks read
        // as zero: they only meet discarded rows or K past the end.  Handling a
        // whole operand stage per pass pays the barrier round trips once per
        // 256 K on wide stages.
        constexpr int H = C::HALVES;
        constexpr int L = (H == 2) ? 2 : 4;
        static_assert(L < FS, "scale lookahead");
        const int KW = (c.KS + H - 1) / H;
        const int total = my_tiles * KW;
        // issue side (entry it)
        int ii = -1, iks = KW;              // tile / stage-in-tile of the next issue
        int is = 0;
        uint32_t iph = 0;
        const float *pa = nullptr, *pb = nullptr;   // this lane's K-block 0 scale of the tile
        bool a_in = false, b_in = false;
        // build side (entry it - L)
        int bi = -1, bks = KW, bs = 0;
        uint32_t bph = 0;
        bool promote = false;
        int bnb = NBB;   // per-row lines: column blocks of the build tile inside N
        bool ok = true;
        // each iteration first releases entry it - L, then issues entry it: the
        // release then finds no copy just issued still in flight
        for (int it = 0; it < total + L && ok; ++it) {
            if (it >= L) {
                if (++bks >= KW) {   // next tile: its path
                    bks = 0;
                    ++bi;
                    const int v = bi & 1;
                    ok = __all_sync(FULL, wait_bar(&ctl->vfull[v], static_cast<uint32_t>(bi >> 1) & 1u, ctl, c));
                    if (!ok) break;
                    promote = ctl->verdict[v] != 0;
                    if constexpr (C::ROWA) bnb = min(NBB, c.N / 32 - sch.tile(unit + bi * nunits).n0 / 32);
                }
                if (lane == 0) trace_event(c, TR_SCALE_BUILD, it - L);
                ok = __all_sync(FULL, wait_bar(&ctl->scfull[bs], bph, ctl, c));
                if (!ok) break;
                if (lane == 0) trace_event(c, TR_SCALE_FULL, it - L);
                if (!promote) {
                    // 8 identical 16-byte lines per 128 rows and half (tcgen05.cp
                    // reads them four times); word w of a line = row (column) block
                    // w, byte j = K block j of the half.
                    uint32_t wa[H], wb[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float *sc = sm_sc + bs * C::SC_ENTRY + h * C::SC_FLOATS;
                        // (per-row / per-column scales: unit lines, 2^0)
                        const float va = (lane < 16 && SK == SCALE_BLOCK32) ? sc[(lane & 3) * 4 + (lane >> 2)] : 1.0f;
                        const float vb = (lane < 4 * NBB && SK != SCALE_ROWCOL) ? sc[16 + (lane & 3) * NBB + (lane >> 2)] : 1.0f;
                        // per-token native tiles have no verdict scan: B's block scales
                        // inside the matrix are checked here
                        if (C::ROWA && (lane >> 2) < bnb && (bks * H + h) * KB_PER_STAGE + (lane & 3) < c.KB &&
                            !is_pow2_scale(vb))
                            atomicOr(c.status, STATUS_SCALE);
                        wa[h] = ue8m0_of(va) << (8 * (lane & 3));
                        wb[h] = ue8m0_of(vb) << (8 * (lane & 3));
                    }
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        wa[h] |= __shfl_xor_sync(FULL, wa[h], 1);
                        wb[h] |= __shfl_xor_sync(FULL, wb[h], 1);
                    }
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        wa[h] |= __shfl_xor_sync(FULL, wa[h], 2);
                        wb[h] |= __shfl_xor_sync(FULL, wb[h], 2);
                    }
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        uint8_t *sf = sm_sf + bs * C::SF_ENTRY + h * C::SF_BYTES;
                        uint4 la;
                        la.x = __shfl_sync(FULL, wa[h], 0);
                        la.y = __shfl_sync(FULL, wa[h], 4);
                        la.z = __shfl_sync(FULL, wa[h], 8);
                        la.w = __shfl_sync(FULL, wa[h], 12);
                        if (!C::ROWA && lane < 8) *reinterpret_cast<uint4 *>(sf + lane * 16) = la;   // (per-row lines: warp 2)
#pragma unroll
                        for (int q = 0; q < C::SFB_CHUNKS; ++q) {
                            uint4 lb;
                            lb.x = __shfl_sync(FULL, wb[h], 16 * q + 0);
                            lb.y = __shfl_sync(FULL, wb[h], 16 * q + 4);
                            lb.z = __shfl_sync(FULL, wb[h], 16 * q + 8);
                            lb.w = __shfl_sync(FULL, wb[h], 16 * q + 12);
                            if (lane < 8) *reinterpret_cast<uint4 *>(sf + C::SF_SET_A + C::SF_SET * q + lane * 16) = lb;
                        }
                    }
                    // the lines become visible to tcgen05.cp's async-proxy reads
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    // (a pair's peer forwards this to the leader from its MMA warp,
                    // which has no copies in flight to wait for)
                    mbar_arrive(&ctl->sfready[bs]);
                    trace_event(c, TR_SCALE_READY, it - L);
                    if (bks == KW - 1) mbar_arrive(&ctl->vempty[bi & 1]);
                }
                __syncwarp();
                if (++bs == FS) { bs = 0; bph ^= 1u; }
            }
            if (it < total) {
                if (++iks >= KW) {   // next tile: per-lane source pointers
                    iks = 0;
                    ++ii;
                    const Tile tt = sch.tile(unit + ii * nunits);
                    const GroupEntry e = sch.entry(tt.g);
                    const int mb = (tt.m0 + row_off) / 32 + (lane >> 2);
                    const int nb = tt.n0 / 32 + (lane >> 2);
                    // (per-row sA: read by the epilogue or by warp 2)
                    a_in = lane < 16 && mb < (tt.Mg + 31) / 32 && SK != SCALE_TOKEN && SK != SCALE_TOKEN_E8;
                    b_in = lane < 4 * NBB && nb < c.N / 32;
                    pa = e.sA + (a_in ? static_cast<int64_t>(mb) * c.KB + (lane & 3) : 0);
                    pb = e.sB + (b_in ? static_cast<int64_t>(nb) * c.KB + (lane & 3) : 0);
                }
                ok = __all_sync(FULL, wait_bar(&ctl->sfempty[is], iph ^ 1u, ctl, c));
                if (!ok) break;
                if (lane == 0) trace_event(c, TR_SCALE_ISSUE, it);
                if constexpr (SK == SCALE_ROWCOL) {
                    mbar_arrive(&ctl->scfull[is]);   // nothing to stage: unit block scales
                } else {
                    const uint32_t sc = smem_u32(sm_sc + is * C::SC_ENTRY);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const int kb = (iks * H + h) * KB_PER_STAGE;   // first K block of the half
                        const bool kb_ok = kb + (lane & 3) < c.KB;
                        const bool ca = a_in && kb_ok, cb = b_in && kb_ok;
                        if (lane < 16) cp_async_4(sc + 4 * (h * C::SC_FLOATS + (lane & 3) * 4 + (lane >> 2)), ca ? pa + kb : pa, ca ? 4u : 0u);
                        if (lane < 4 * NBB)
                            cp_async_4(sc + 4 * (h * C::SC_FLOATS + 16 + (lane & 3) * NBB + (lane >> 2)), cb ? pb + kb : pb, cb ? 4u : 0u);
                    }
                    cp_async_mbar_arrive_noinc(&ctl->scfull[is]);
                }
                if (++is == FS) { is = 0; iph ^= 1u; }
            }
        }
        // no scale copy may still be landing when the CTA exits
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ epilogue / promotion
        const int q = warp & 3;                       // tensor-memory lane quarter
        const int h = (warp - EPI_WARP0) >> 2;        // column half
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        constexpr int NCH = C::EPI_COLS / 32;         // 32-column chunks per warp
        uint32_t uses0 = 0, uses1 = 0, pk = 0;
        int eft = 0;   // scale-ring entries of the tiles before this one
        // Single problems write native tiles through shared memory with TMA
        // stores: one lane per output row would otherwise flood the load/store
        // path with row-scattered stores for thousands of cycles, and the MMA
        // thread's barrier operations queue behind them.  The four warps of a
        // column half share a staging buffer and a named barrier; every exit
        // from the loop is agreed among them first (named_bar_and), so no warp
        // is ever left waiting at that barrier.  A promotion tile agrees once,
        // after its K loop: a warp whose wait failed skips the rest of the loop
        // and the others' waits end on the abort flag, so all reach that point
        // (agreeing per K block would hold the four warps in lockstep).
        constexpr bool TMA_OUT = !GROUPED;
        const uint32_t bar_id = 1u + static_cast<uint32_t>(h);
        constexpr uint32_t HALF_THREADS = 128;
        const bool issuer = q == 0 && lane == 0;
        uint32_t rph = 0;             // residual chunks loaded for this column half (rfull phase)
        bool r_pending = false;       // issuer: a residual load may still be landing
        for (int i = 0; i < my_tiles; ++i) {
            const int v = i & 1;
            bool ok = wait_bar(&ctl->vfull[v], static_cast<uint32_t>(i >> 1) & 1u, ctl, c);
            ok = __all_sync(FULL, ok);
            if constexpr (TMA_OUT) ok = named_bar_and(bar_id, HALF_THREADS, ok);
            if (!ok) break;
            const bool promote = ctl->verdict[v] != 0;
            const Tile tt = sch.tile(unit + i * nunits);
            const GroupEntry e = sch.entry(tt.g);
            const int row = tt.m0 + row_off + 32 * q + lane;
            // (grouped tiles own only the first TILE_M of the MMA's 128 rows)
            const bool row_ok = row < tt.Mg && 32 * q + lane < C::TILE_M;
            const int col0 = h * C::EPI_COLS;
            __nv_bfloat16 *crow = e.C + static_cast<int64_t>(row_ok ? row : 0) * c.N + tt.n0;
            if constexpr (RES) {
                // this thread's 256 bytes of the residual row into L2 while the
                // tile's K loop runs: the chunk loads of the epilogue (and the
                // last tile's, which nothing overlaps) then hit L2 (+1 % on the
                // 4096^3 GEMM with a residual)
                if (row_ok) {
                    const __nv_bfloat16 *rr = args.R + static_cast<int64_t>(row) * c.N + tt.n0 + col0;
                    if (tt.n0 + col0 < c.N) prefetch_l2(rr);
                    if (tt.n0 + col0 + 64 < c.N) prefetch_l2(rr + 64);
                }
            }

            if (!promote) {
                // One warp per column half polls for the accumulator: the one of lane
                // quarter 0, whose sub-partition the MMA thread does not share; the
                // half's other warps wait in its named barrier.  Polling warps beside
                // the MMA thread slow its issue (4-6 % on the prefill GEMM).
                if (!TMA_OUT || q == 0) ok = __all_sync(FULL, wait_poll(&ctl->tfull[0], uses0 & 1u, ctl, c));
                if constexpr (TMA_OUT) ok = named_bar_and(bar_id, HALF_THREADS, ok);
                if (!ok) break;
                if (warp == EPI_WARP0 && lane == 0) trace_event(c, TR_EPI_FULL, i);
                tc_fence_after();
                // drain the whole accumulator slice, then release it at once
                uint32_t r[NCH][32];
#pragma unroll
                for (int x = 0; x < NCH; ++x) tmem_ld_x32(tmem + lane_base + col0 + 32 * x, r[x]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // the loads above have completed (tcgen05.wait::ld), so the
                    // leader may overwrite the accumulator: a plain signal suffices
                    mbar_arrive(&ctl->tempty[0]);
                    if (PAIR && !leader) mbar_signal_cluster(mapa_shared(&ctl->tempty[0], 0));
                }
                if (warp == EPI_WARP0 && lane == 0) trace_event(c, TR_EPI_RELEASED, i);
                ++uses0;
                if constexpr (TMA_OUT) {
                    // 32-column chunks: rows into the half's staging buffer, then
                    // one TMA store of the 128 x 32 box (rows past M are clipped)
                    __nv_bfloat16 *stg = sm_stg + h * (BM * C::STG_COLS);
                    uint4 *mine = reinterpret_cast<uint4 *>(stg + (32 * q + lane) * C::STG_COLS);
                    // per-row / per-column scales: this thread's row factor
                    const float rs = (SK == SCALE_ROWCOL && row_ok) ? __ldg(e.sA + row) : 1.0f;
#pragma unroll
                    for (int x = 0; x < NCH; ++x) {
                        if (SK == SCALE_ROWCOL && tt.n0 + col0 + 32 * x < c.N) {
                            const float *cs = e.sB + tt.n0 + col0 + 32 * x;   // 32 column factors (broadcast)
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                r[x][j] = __float_as_uint(__uint_as_float(r[x][j]) * (rs * __ldg(cs + j)));
                        }
                        if constexpr (RES) {
                            {
                                // the residual chunk comes into the staging buffer by TMA
                                // first (rows past M read as zero); each thread adds its row
                                const int col = tt.n0 + col0 + 32 * x;
                                if (issuer) {
                                    if (col < c.N) {
                                        mbar_arrive_expect_tx(&ctl->rfull[h], BM * C::STG_COLS * 2);
                                        tma_load_2d(&args.tmR, &ctl->rfull[h], stg, col, tt.m0 + row_off);
                                        r_pending = true;
                                    } else {
                                        mbar_arrive(&ctl->rfull[h]);   // keeps the phase sequence
                                    }
                                }
                                bool rok = __all_sync(FULL, wait_bar(&ctl->rfull[h], rph & 1u, ctl, c));
                                rok = named_bar_and(bar_id, HALF_THREADS, rok);   // the half leaves together
                                ++rph;
                                if (!rok) {
                                    ok = false;
                                    break;
                                }
                                if (issuer) r_pending = false;
                                add_bf16x32(r[x], mine);
                            }
                        }
                        if constexpr (QOUT) {
                            // the warp's 32 rows x these 32 columns are one 32 x 32 block:
                            // bf16, block scale, codes; the codes go out by TMA as a
                            // 128 x 32-byte box, the scale by lane 0
                            uint32_t bw[16], cd[8];
                            bf16_words32(bw, r[x], row_ok);
                            const float sc = quantize_rows32(bw, cd);
                            uint4 *qm = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(stg) + (32 * q + lane) * 32);
                            qm[0] = make_uint4(cd[0], cd[1], cd[2], cd[3]);
                            qm[1] = make_uint4(cd[4], cd[5], cd[6], cd[7]);
                            const int col = tt.n0 + col0 + 32 * x;
                            const int rb0 = tt.m0 + row_off + 32 * q;   // the block's first row
                            if (lane == 0 && col < c.N && rb0 < c.M)
                                args.sC[static_cast<int64_t>(rb0 / 32) * (c.N / 32) + col / 32] = sc;
                        } else {
                            pack_bf16x32(mine, r[x]);
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(bar_id, HALF_THREADS);
                        if (issuer) {
                            const int col = tt.n0 + col0 + 32 * x;
                            if (col < c.N) {
                                if constexpr (QOUT) tma_store_2d(&args.tmQ, stg, col, tt.m0 + row_off);
                                else tma_store_2d(&args.tmC, stg, col, tt.m0 + row_off);
                                bulk_commit_group();
                                bulk_wait_read_all();
                            }
                        }
                        named_bar_sync(bar_id, HALF_THREADS);   // the buffer is free again
                    }
                    if (!ok) break;
                } else if (row_ok) {
#pragma unroll
                    for (int x = 0; x < NCH; ++x)
                        if (tt.n0 + col0 + 32 * x < c.N) store_bf16x32(crow + col0 + 32 * x, r[x]);
                }
                if (warp == EPI_WARP0 && lane == 0) trace_event(c, TR_EPI_STORED, i);
            } else {
                if (pk & 1u) ++pk;
                // Each K block's scales come from the stage's scale-ring entry
                // (the MMA warp releases an entry only after every partial of
                // its stage has been read here): row block q of this CTA, the
                // warp's NCH column blocks.
                int f = eft % FS, hh = 0, j = 0;
                uint32_t fph = static_cast<uint32_t>(eft / FS) & 1u;
                float acc[C::EPI_COLS];
#pragma unroll
                for (int x = 0; x < C::EPI_COLS; ++x) acc[x] = 0.0f;
                for (int kb = 0; kb < c.KB; ++kb) {
                    const uint32_t b = pk & 1u;
                    const uint32_t ub = b ? uses1 : uses0;
                    if (hh == 0 && j == 0) {   // a new stage: its entry has landed
                        ok = __all_sync(FULL, wait_bar(&ctl->sfready[f], fph, ctl, c));
                        if (!ok) break;
                    }
                    // scale products sA * sB of this K block, one per 32-column block
                    const float *se = sm_sc + f * C::SC_ENTRY + hh * C::SC_FLOATS;
                    static_assert(NCH == 4, "one 16-byte load of column scales per K block");
                    float sa;
                    if constexpr (SK == SCALE_TOKEN) sa = row_ok ? __ldg(e.sA + static_cast<int64_t>(row) * c.KB + kb) : 0.0f;
                    else sa = se[j * 4 + q];
                    const float4 sb = *reinterpret_cast<const float4 *>(se + 16 + j * NBB + h * NCH);
                    const float sc[NCH] = {sa * sb.x, sa * sb.y, sa * sb.z, sa * sb.w};
                    if (++j == KB_PER_STAGE) {
                        j = 0;
                        if (++hh == C::HALVES) {
                            hh = 0;
                            if (++f == FS) { f = 0; fph ^= 1u; }
                        }
                    }
                    ok = __all_sync(FULL, wait_bar(&ctl->tfull[b], ub & 1u, ctl, c));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pbase = tmem + lane_base + b * BN + col0;
#pragma unroll
                    for (int x = 0; x < 2 * NCH; ++x) {
                        uint32_t r[16];
                        tmem_ld_x16(pbase + 16 * x, r);
                        tmem_ld_wait();
                        if (x == 2 * NCH - 1) {
                            tc_fence_before();
                            __syncwarp();
                            // (a pair's peer: its MMA warp forwards the release)
                            if (lane == 0) mbar_arrive(&ctl->tempty[b]);
                        }
                        if constexpr (PAIR) {
#pragma unroll
                            for (int y = 0; y < 16; ++y)
                                acc[16 * x + y] = fmaf(sc[x >> 1], __uint_as_float(r[y]), acc[16 * x + y]);
                        } else {
                            // single-CTA tiles: packed two-lane FMAs (the same fma per
                            // element, half the issue slots; measured 6 % faster here,
                            // not on CTA pairs)
                            const uint64_t s2 = f32x2_pack(__float_as_uint(sc[x >> 1]), __float_as_uint(sc[x >> 1]));
#pragma unroll
                            for (int y = 0; y < 8; ++y) {
                                uint64_t a2 = f32x2_pack(__float_as_uint(acc[16 * x + 2 * y]),
                                                         __float_as_uint(acc[16 * x + 2 * y + 1]));
                                fma_f32x2(a2, s2, f32x2_pack(r[2 * y], r[2 * y + 1]));
                                uint32_t lo, hi;
                                f32x2_unpack(a2, lo, hi);
                                acc[16 * x + 2 * y] = __uint_as_float(lo);
                                acc[16 * x + 2 * y + 1] = __uint_as_float(hi);
                            }
                        }
                    }
                    if (b) ++uses1; else ++uses0;
                    ++pk;
                }
                if constexpr (TMA_OUT) ok = named_bar_and(bar_id, HALF_THREADS, ok);
                if (!ok) break;
                if constexpr (QOUT) {
                    // every lane takes part in each block's maximum; codes and
                    // scales go out by plain stores
#pragma unroll
                    for (int x = 0; x < NCH; ++x) {
                        uint32_t bw[16], cd[8];
                        bf16_words32f(bw, acc + 32 * x, row_ok);
                        const float sc = quantize_rows32(bw, cd);
                        const int col = tt.n0 + col0 + 32 * x;
                        const int rb0 = tt.m0 + row_off + 32 * q;
                        if (col < c.N) {
                            if (row_ok) {
                                uint4 *dq = reinterpret_cast<uint4 *>(args.Cq + static_cast<int64_t>(row) * c.N + col);
                                dq[0] = make_uint4(cd[0], cd[1], cd[2], cd[3]);
                                dq[1] = make_uint4(cd[4], cd[5], cd[6], cd[7]);
                            }
                            if (lane == 0 && rb0 < c.M)
                                args.sC[static_cast<int64_t>(rb0 / 32) * (c.N / 32) + col / 32] = sc;
                        }
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int x = 0; x < NCH; ++x) {
                        if (tt.n0 + col0 + 32 * x >= c.N) continue;
                        if constexpr (RES) {
                            {   // residual of this row (16-byte loads)
                                const uint4 *rr = reinterpret_cast<const uint4 *>(
                                    args.R + static_cast<int64_t>(row) * c.N + tt.n0 + col0 + 32 * x);
#pragma unroll
                                for (int w = 0; w < 4; ++w) {
                                    const uint4 u = __ldg(rr + w);
                                    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                                    for (int k = 0; k < 4; ++k) {
                                        acc[32 * x + 8 * w + 2 * k] += __uint_as_float(wv[k] << 16);
                                        acc[32 * x + 8 * w + 2 * k + 1] += __uint_as_float(wv[k] & 0xFFFF0000u);
                                    }
                                }
                            }
                        }
                        store_bf16x32f(crow + col0 + 32 * x, acc + 32 * x);
                    }
                }
            }
            eft += (c.KS + C::HALVES - 1) / C::HALVES;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->vempty[v]);
        }
        if (TMA_OUT && issuer) {
            // no residual load may still be landing, and the output is written,
            // before the CTA exits
            if (r_pending) wait_bar_drain(&ctl->rfull[h], (rph - 1u) & 1u, c.wait_limit);
            bulk_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
        else tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BN, int SK = SCALE_BLOCK32>
__global__ void __launch_bounds__(NUM_THREADS, 1) bsfp8_gemm_plain(const __grid_constant__ PlainArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, false, false, PlainArgs, SK>(args, smem_raw);
}

// CTA-pair variant: clusters of two CTAs, 256-row tiles, pair MMAs.
template <int BN, int SK = SCALE_BLOCK32, bool RES = false, bool QOUT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    bsfp8_gemm_pair(const __grid_constant__ PlainArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, false, true, PlainArgs, SK, RES, QOUT>(args, smem_raw);
}

template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1) bsfp8_gemm_grouped(const __grid_constant__ GroupedArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, true, false>(args, smem_raw);
}

// Grouped problems with device-resident records (one warp per group): checks
// the record (no null pointer; A, B, C 16-byte and sA, sB 4-byte aligned),
// writes the group's B tensor map -- the host-encoded template (shape N x K,
// box of BN rows) with the record's B as its base -- into maps[g], and
// valid[g].  A rejected record sets STATUS_RECORD; its group is skipped.
__global__ void __launch_bounds__(128) bsfp8_grouped_prepare(const __grid_constant__ CUtensorMap tmpl,
                                                            const GroupRecord *table, int G, CUtensorMap *maps,
                                                            int32_t *valid, uint32_t *status) {
    __shared__ alignas(128) CUtensorMap sm_map[4];
    const int w = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int g = static_cast<int>(blockIdx.x) * 4 + w;
    if (g >= G) return;   // the whole warp
    if (lane < 8) reinterpret_cast<uint4 *>(&sm_map[w])[lane] = reinterpret_cast<const uint4 *>(&tmpl)[lane];
    const GroupRecord r = table[g];
    const auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
    const bool ok = r.A && r.sA && r.B && r.sB && r.C && al(r.A, 16) && al(r.B, 16) && al(r.C, 16) &&
                    al(r.sA, 4) && al(r.sB, 4);
    __syncwarp();
    if (ok) {
        if (lane == 0) tensormap_set_base_smem(smem_u32(&sm_map[w]), reinterpret_cast<uint64_t>(r.B));
        __syncwarp();
        tensormap_publish(&maps[g], smem_u32(&sm_map[w]));
    }
    if (lane == 0) {
        valid[g] = ok ? 1 : 0;
        if (!ok) atomicOr(status, STATUS_RECORD);
    }
}

template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1) bsfp8_gemm_grouped_dev(const __grid_constant__ GroupedDevArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, true, false>(args, smem_raw);
}

// C = 0 for K == 0 (an empty sum).
__global__ void bsfp8_zero_fill(uint4 *p, int64_t n16) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void bsfp8_fill_f32(float *p, float v, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

}  // namespace bsfp8

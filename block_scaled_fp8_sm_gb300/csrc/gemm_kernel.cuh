// gemm_kernel.cuh -- persistent, warp-specialised block-scaled E4M3 GEMM for
// sm_103a (tcgen05 tensor cores, tensor memory accumulators, TMA).
//
// Computes C[m,n] = bf16( sum_kb sA[m/32][kb] * sB[n/32][kb] * sum_{k in kb}
// A[m,k] B[n,k] ) (FP8 GEMM library article, hncyxsy.com/news/241433,
// sections 2.2-2.3: 32x32 block scales that take part in the accumulation),
// for one problem or for a group of independent problems (same article,
// section 4.2: one launch, each block looks up its problem in a table).
//
// Roles (384 threads, one CTA per SM, persistent over output tiles):
//   warp 0     producer: TMA loads of the A and B K-slices into a ring of
//              shared-memory stages (128-byte swizzle; for grouped problems A
//              rows come by cp.async since the row counts live on the device),
//              plus the stage's scale lines: the 32x32 block scales of the
//              tile converted to UE8M0 bytes in the layout tcgen05.cp wants.
//   warp 1     MMA issuer (one thread): native path = tcgen05.mma
//              kind::mxf8f6f4 with the UE8M0 scales copied into tensor memory;
//              promotion path = one unscaled kind::f8f6f4 MMA per 32-K block
//              into a fresh tensor-memory partial.
//   warp 2     path verdict: scans each tile's scales one or two tiles ahead
//              and decides native (all positive normal powers of two) or
//              promotion.
//   warps 4-11 epilogue: tensor memory -> registers -> bf16 -> global
//              (native); or per-32-K-block promotion acc += sA*sB*partial in
//              fp32 registers, then bf16 -> global.
//
// The K loop of every tile runs whole and in ascending K order, with a tile
// shape that depends only on (N, grouped or not): no split-K, no stream-K, so
// each output row is independent of M and of the other rows ("AI Infra
// 进阶：如何让大模型输出确定的结果", aif.amtbbs.org post 29992, section 1).
//
// Every wait is bounded (clock64 budget).  On expiry a CTA-wide abort flag
// and the device status word are set, every role leaves its loop, in-flight
// TMA loads and MMAs are drained with bounded waits, tensor memory is freed
// and the kernel returns.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace bsfp8 {

constexpr int BM = 128;            // rows of A per tile (MMA M)
constexpr int BK = 128;            // K elements (= bytes) per pipeline stage
constexpr int KB_PER_STAGE = 4;    // 32-K scale blocks per stage
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int MAX_GROUPS = 64;
constexpr int GROUP_M = 8;         // tile-order swizzle width (m-tiles) for L2 reuse

enum : uint32_t { STATUS_TIMEOUT = 1u, STATUS_SCALE = 2u };
enum : int { PATH_AUTO = 0, PATH_NATIVE = 1, PATH_PROMOTE = 2 };

template <int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SFB_CHUNKS = (BN + 127) / 128;           // 128 B rows per tcgen05.cp
    static constexpr int SF_BYTES = 512 * (1 + SFB_CHUNKS);         // scale lines per stage
    static constexpr int SF_COLS = 4 * (1 + SFB_CHUNKS);            // tensor-memory columns per stage
    static constexpr int ACC_COLS = 2 * BN;                         // two accumulator / partial buffers
    static constexpr int SF_COL0 = ACC_COLS;
    static constexpr int TMEM_USED = ACC_COLS + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
    static constexpr int EPI_COLS = BN / 2;                         // columns per epilogue warp
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
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
};

struct PlainArgs {
    CUtensorMap tmA;
    CUtensorMap tmB;
    GroupEntry e;
    Common c;
};

struct GroupedArgs {
    CUtensorMap tmB[MAX_GROUPS];
    GroupEntry e[MAX_GROUPS];
    Common c;
};

template <int STAGES>
struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t vfull[2];
    uint64_t vempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int verdict[2];
    int abort;
    int num_tiles;
    int tile_start[MAX_GROUPS + 1];
    int mg[MAX_GROUPS];
};

struct Tile {
    int m0, n0, Mg, g;
};

template <int BN>
constexpr int smem_bytes() {
    using C = Cfg<BN>;
    return 1024 + C::STAGES * (C::A_BYTES + C::B_BYTES + C::SF_BYTES) +
           static_cast<int>(sizeof(Ctrl<C::STAGES>));
}

// ---------------------------------------------------------------------------
template <int STAGES>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Ctrl<STAGES> *ctl,
                                         const Common &c) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
        if (clock64() - t0 > c.wait_limit) {
            *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
            atomicOr(c.status, STATUS_TIMEOUT);
            return false;
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

template <int BN, bool GROUPED, typename Args>
struct Sched {
    const Args &a;
    const Common &c;
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
            r.m0 = (first_m + in % gsz) * BM;
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
            const int mtg = (Mg + BM - 1) / BM;
            const int local = t - tile_start[g];
            r.m0 = (local % mtg) * BM;
            r.n0 = (local / mtg) * BN;
            r.Mg = Mg;
            r.g = g;
        }
        return r;
    }

    __device__ __forceinline__ const GroupEntry &entry(int g) const {
        if constexpr (!GROUPED) return a.e;
        else return a.e[g];
    }
};

// Scales of one pipeline stage as this lane holds them: lane l < 16 carries
// sA[row block l/4][kb l%4], lane l < 4*BN/32 carries sB[row block l/4][kb l%4].
// Absent blocks read as 1.0 (UE8M0 127): they only meet zero-filled or
// discarded rows.
template <int BN, bool GROUPED, typename S>
__device__ __forceinline__ void load_stage_scales(const S &sch, int j, int total, int lane,
                                                  float &va, float &vb) {
    va = 1.0f;
    vb = 1.0f;
    if (j >= total) return;
    const Common &c = sch.c;
    const Tile tt = sch.tile(blockIdx.x + (j / c.KS) * gridDim.x);
    const GroupEntry &e = sch.entry(tt.g);
    const int kb = (j % c.KS) * KB_PER_STAGE + (lane & 3);
    if (kb >= c.KB) return;
    const int MB = (tt.Mg + 31) / 32;
    if (lane < 16) {
        const int mb = tt.m0 / 32 + (lane >> 2);
        if (mb < MB) va = __ldg(e.sA + static_cast<int64_t>(mb) * c.KB + kb);
    }
    if (lane < 4 * (BN / 32)) {
        const int nb = tt.n0 / 32 + (lane >> 2);
        if (nb < c.N / 32) vb = __ldg(e.sB + static_cast<int64_t>(nb) * c.KB + kb);
    }
}

__device__ __forceinline__ uint32_t ue8m0_of(float v) { return (__float_as_uint(v) >> 23) & 0xFFu; }

// ---------------------------------------------------------------------------
template <int BN, bool GROUPED, typename Args>
__device__ __forceinline__ void gemm_body(const Args &args, uint8_t *smem_raw) {
    using C = Cfg<BN>;
    constexpr int S = C::STAGES;
    constexpr uint32_t FULL = 0xFFFFFFFFu;
    const Common &c = args.c;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::A_BYTES;
    uint8_t *sm_sf = sm_b + S * C::B_BYTES;
    Ctrl<S> *ctl = reinterpret_cast<Ctrl<S> *>(sm_sf + S * C::SF_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], NUM_EPI_WARPS);
            mbar_init(&ctl->vfull[b], 1);
            mbar_init(&ctl->vempty[b], 1 + NUM_EPI_WARPS);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) {
        if constexpr (GROUPED) {
            // tile table: group g owns tiles [tile_start[g], tile_start[g+1])
            if (lane == 0) {
                int acc = 0;
                for (int g = 0; g < c.G; ++g) {
                    int m = c.Ms[g];
                    m = m < 0 ? 0 : m;
                    ctl->mg[g] = m;
                    ctl->tile_start[g] = acc;
                    acc += ((m + BM - 1) / BM) * c.nt;
                }
                ctl->tile_start[c.G] = acc;
                ctl->num_tiles = acc;
            }
        } else {
            if (lane == 0) ctl->num_tiles = c.num_tiles;
        }
    }
    if (warp == 0 && lane == 0) {
        if constexpr (!GROUPED) {
            tma_prefetch_desc(&args.tmA);
            tma_prefetch_desc(&args.tmB);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = ctl->tmem_base;
    const int num_tiles = ctl->num_tiles;
    const int my_tiles =
        (static_cast<int>(blockIdx.x) < num_tiles)
            ? (num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                  static_cast<int>(gridDim.x)
            : 0;
    const Sched<BN, GROUPED, Args> sch{args, c, ctl->tile_start, ctl->mg};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // grouped problems: the cp.async A rows of a stage are waited for D
        // iterations later, so D stages of copies are in flight while the MMA
        // may run up to S-D stages behind the producer.
        constexpr int D = S / 2;
        const int total = my_tiles * c.KS;
        float pa0, pb0, pa1, pb1, pa2, pb2, pa3, pb3;
        load_stage_scales<BN, GROUPED>(sch, 0, total, lane, pa0, pb0);
        load_stage_scales<BN, GROUPED>(sch, 1, total, lane, pa1, pb1);
        load_stage_scales<BN, GROUPED>(sch, 2, total, lane, pa2, pb2);
        load_stage_scales<BN, GROUPED>(sch, 3, total, lane, pa3, pb3);
        int withheld = -1;   // slot never armed (test hook), excluded from the drain
        int it = 0;
        bool ok = true;
        for (; it < total; ++it) {
            const int s = it % S;
            const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
            ok = wait_bar(&ctl->empty[s], ph ^ 1u, ctl, c);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            const int ti = it / c.KS;
            const int ks = it % c.KS;
            const Tile tt = sch.tile(static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x));
            const int k0 = ks * BK;
            const bool withhold = (c.withhold_stage == it) && blockIdx.x == 0;
            if (withhold) {
                withheld = s;
            } else {
                // full[s] counts one arrival: the transaction bytes are registered
                // first, the arrival comes once the scale lines (and, for grouped
                // problems, the cp.async A rows) are in shared memory.
                if (lane == 0) {
                    if constexpr (!GROUPED) {
                        mbar_expect_tx(&ctl->full[s], C::A_BYTES + C::B_BYTES);
                        tma_load_2d(&args.tmA, &ctl->full[s], sm_a + s * C::A_BYTES, k0, tt.m0);
                        tma_load_2d(&args.tmB, &ctl->full[s], sm_b + s * C::B_BYTES, k0, tt.n0);
                    } else {
                        mbar_expect_tx(&ctl->full[s], C::B_BYTES);
                        tma_load_2d(&args.tmB[tt.g], &ctl->full[s], sm_b + s * C::B_BYTES, k0, tt.n0);
                    }
                }
                // scale lines for this stage (UE8M0, 32 identical 16-byte lines per chunk)
                uint32_t wa = ue8m0_of(pa0) << (8 * (lane & 3));
                wa |= __shfl_xor_sync(FULL, wa, 1);
                wa |= __shfl_xor_sync(FULL, wa, 2);
                uint32_t wb = ue8m0_of(pb0) << (8 * (lane & 3));
                wb |= __shfl_xor_sync(FULL, wb, 1);
                wb |= __shfl_xor_sync(FULL, wb, 2);
                uint4 la;
                la.x = __shfl_sync(FULL, wa, 0);
                la.y = __shfl_sync(FULL, wa, 4);
                la.z = __shfl_sync(FULL, wa, 8);
                la.w = __shfl_sync(FULL, wa, 12);
                uint8_t *sf = sm_sf + s * C::SF_BYTES;
                *reinterpret_cast<uint4 *>(sf + lane * 16) = la;
#pragma unroll
                for (int q = 0; q < C::SFB_CHUNKS; ++q) {
                    uint4 lb;
                    lb.x = __shfl_sync(FULL, wb, 16 * q + 0);
                    lb.y = __shfl_sync(FULL, wb, 16 * q + 4);
                    lb.z = __shfl_sync(FULL, wb, 16 * q + 8);
                    lb.w = __shfl_sync(FULL, wb, 16 * q + 12);
                    *reinterpret_cast<uint4 *>(sf + 512 * (1 + q) + lane * 16) = lb;
                }
                if constexpr (GROUPED) {
                    // A rows of this group: 16-byte cp.async into the swizzled layout;
                    // chunks past K are zero-filled, rows past M_g are not loaded
                    // (they only feed output rows that are never stored).
                    const GroupEntry &e = sch.entry(tt.g);
                    const int rows = min(BM, tt.Mg - tt.m0);
                    const uint32_t dst0 = smem_u32(sm_a + s * C::A_BYTES);
                    for (int idx = lane; idx < rows * 8; idx += 32) {
                        const int r = idx >> 3, ch = idx & 7;
                        const int kk = k0 + ch * 16;
                        const bool in = kk < c.K;
                        const uint8_t *src =
                            e.A + static_cast<int64_t>(tt.m0 + r) * c.K + (in ? kk : 0);
                        const uint32_t dst = dst0 + r * 128 + ((ch ^ (r & 7)) << 4);
                        cp_async_16(dst, src, in ? 16u : 0u);
                    }
                    cp_async_commit();
                }
                if constexpr (!GROUPED) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->full[s]);
                } else {
                    // arrive for the stage issued D iterations ago once its copies landed
                    cp_async_wait_group<D>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    const int old = it - D;
                    if (old >= 0 && lane == 0 && (old % S) != withheld) mbar_arrive(&ctl->full[old % S]);
                }
            }
            if constexpr (GROUPED) {
                if (withhold) {
                    cp_async_commit();   // keep one group per iteration
                    cp_async_wait_group<D>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    const int old = it - D;
                    if (old >= 0 && lane == 0 && (old % S) != withheld) mbar_arrive(&ctl->full[old % S]);
                }
            }
            pa0 = pa1; pb0 = pb1;
            pa1 = pa2; pb1 = pb2;
            pa2 = pa3; pb2 = pb3;
            load_stage_scales<BN, GROUPED>(sch, it + 4, total, lane, pa3, pb3);
        }
        if constexpr (GROUPED) {
            // stages whose arrive is still pending: those issued in the last S-1 iterations
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                for (int old = max(0, it - D); old < it; ++old)
                    if ((old % S) != withheld) mbar_arrive(&ctl->full[old % S]);
            }
        }
        // drain: every armed stage's last phase must complete before the CTA exits
        if (lane == 0) {
            for (int d = max(0, it - S); d < it; ++d) {
                const int s = d % S;
                if (s == withheld && d >= it - S) continue;
                wait_bar_drain(&ctl->full[s], static_cast<uint32_t>(d / S) & 1u, c.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int it = 0;
            uint32_t u = 0;
            bool ok = true;
            bool issued = false;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int v = i & 1;
                ok = wait_bar(&ctl->vfull[v], static_cast<uint32_t>(i >> 1) & 1u, ctl, c);
                if (!ok) break;
                const bool promote = ctl->verdict[v] != 0;
                if (!promote) {
                    const uint32_t buf = u & 1u;
                    ok = wait_bar(&ctl->tempty[buf], ((u >> 1) & 1u) ^ 1u, ctl, c);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + buf * BN;
                    for (int ks = 0; ks < c.KS; ++ks, ++it) {
                        const int s = it % S;
                        ok = wait_bar(&ctl->full[s], static_cast<uint32_t>(it / S) & 1u, ctl, c);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sfa = tmem + C::SF_COL0 + s * C::SF_COLS;
                        const uint32_t sfb = sfa + 4;
                        const uint32_t sf_s = smem_u32(sm_sf + s * C::SF_BYTES);
                        tmem_cp_32x128b_warpx4(sfa, sdesc_sf_lines(sf_s));
#pragma unroll
                        for (int q = 0; q < C::SFB_CHUNKS; ++q)
                            tmem_cp_32x128b_warpx4(sfb + 4 * q, sdesc_sf_lines(sf_s + 512 * (1 + q)));
                        const uint64_t ad = sdesc_k_sw128(smem_u32(sm_a + s * C::A_BYTES));
                        const uint64_t bd = sdesc_k_sw128(smem_u32(sm_b + s * C::B_BYTES));
                        const int nk = min(KB_PER_STAGE, c.KB - ks * KB_PER_STAGE);
                        issued = true;
                        for (int j = 0; j < nk; ++j) {
                            mma_mxf8(d, ad + static_cast<uint64_t>(2 * j), bd + static_cast<uint64_t>(2 * j),
                                     idesc_mxf8f6f4(BM, BN, j, j), sfa, sfb,
                                     (ks | j) != 0 ? 1u : 0u);
                        }
                        mma_commit(&ctl->empty[s]);
                    }
                    if (!ok) break;
                    mma_commit(&ctl->tfull[buf]);
                    ++u;
                } else {
                    for (int ks = 0; ks < c.KS && ok; ++ks, ++it) {
                        const int s = it % S;
                        ok = wait_bar(&ctl->full[s], static_cast<uint32_t>(it / S) & 1u, ctl, c);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t ad = sdesc_k_sw128(smem_u32(sm_a + s * C::A_BYTES));
                        const uint64_t bd = sdesc_k_sw128(smem_u32(sm_b + s * C::B_BYTES));
                        const int nk = min(KB_PER_STAGE, c.KB - ks * KB_PER_STAGE);
                        for (int j = 0; j < nk; ++j) {
                            const uint32_t buf = u & 1u;
                            ok = wait_bar(&ctl->tempty[buf], ((u >> 1) & 1u) ^ 1u, ctl, c);
                            if (!ok) break;
                            tc_fence_after();
                            issued = true;
                            mma_f8(tmem + buf * BN, ad + static_cast<uint64_t>(2 * j),
                                   bd + static_cast<uint64_t>(2 * j), idesc_f8f6f4(BM, BN), 0u);
                            mma_commit(&ctl->tfull[buf]);
                            ++u;
                        }
                        if (!ok) break;
                        mma_commit(&ctl->empty[s]);
                    }
                    if (!ok) break;
                }
                mbar_arrive(&ctl->vempty[v]);
            }
            // all issued tensor-core work must finish before tensor memory is freed
            if (issued) {
                mma_commit(&ctl->drain);
                wait_bar_drain(&ctl->drain, 0u, c.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // -------------------------------------------------------- path verdict
        for (int i = 0; i < my_tiles; ++i) {
            const int v = i & 1;
            bool ok = wait_bar(&ctl->vempty[v], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u, ctl, c);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            int verdict = 1;
            if (c.mode != PATH_PROMOTE) {
                const Tile tt = sch.tile(static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x));
                const GroupEntry &e = sch.entry(tt.g);
                const int MB = (tt.Mg + 31) / 32;
                const int mb0 = tt.m0 / 32, mb1 = min(mb0 + BM / 32, MB);
                const int nb0 = tt.n0 / 32, nb1 = min(nb0 + BN / 32, c.N / 32);
                bool bad = false;
                // each tile's scales are two contiguous row ranges of sA and sB
                const float *pa = e.sA + static_cast<int64_t>(mb0) * c.KB;
                const int na = (mb1 - mb0) * c.KB;
                const float *pb = e.sB + static_cast<int64_t>(nb0) * c.KB;
                const int nbn = (nb1 - nb0) * c.KB;
                for (int x = lane; x < na; x += 32 * 8) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (x + 32 * u < na) bad |= !is_pow2_scale(__ldg(pa + x + 32 * u));
                }
                for (int x = lane; x < nbn; x += 32 * 8) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (x + 32 * u < nbn) bad |= !is_pow2_scale(__ldg(pb + x + 32 * u));
                }
                const bool any_bad = __any_sync(FULL, bad);
                verdict = any_bad ? 1 : 0;
                if (any_bad && c.mode == PATH_NATIVE && lane == 0) atomicOr(c.status, STATUS_SCALE);
            }
            if (lane == 0) {
                ctl->verdict[v] = verdict;
                mbar_arrive(&ctl->vfull[v]);
            }
            __syncwarp();
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ epilogue / promotion
        const int q = warp & 3;                       // tensor-memory lane quarter
        const int h = (warp - EPI_WARP0) >> 2;        // column half
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        uint32_t u = 0;
        for (int i = 0; i < my_tiles; ++i) {
            const int v = i & 1;
            bool ok = wait_bar(&ctl->vfull[v], static_cast<uint32_t>(i >> 1) & 1u, ctl, c);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            const bool promote = ctl->verdict[v] != 0;
            const Tile tt = sch.tile(static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x));
            const GroupEntry &e = sch.entry(tt.g);
            const int row = tt.m0 + 32 * q + lane;
            const bool row_ok = row < tt.Mg;
            const int col0 = h * C::EPI_COLS;
            __nv_bfloat16 *crow = e.C + static_cast<int64_t>(row_ok ? row : 0) * c.N + tt.n0;

            if (!promote) {
                const uint32_t buf = u & 1u;
                ok = wait_bar(&ctl->tfull[buf], (u >> 1) & 1u, ctl, c);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < C::EPI_COLS / 32; ++ch) {
                    uint32_t r[32];
                    const int col = col0 + 32 * ch;
                    tmem_ld_x32(tmem + lane_base + buf * BN + col, r);
                    tmem_ld_wait();
                    if (ch == C::EPI_COLS / 32 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                    }
                    if (row_ok && tt.n0 + col < c.N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint4 o;
                            __nv_bfloat162 p0 = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 0]), __uint_as_float(r[8 * w + 1]));
                            __nv_bfloat162 p1 = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 2]), __uint_as_float(r[8 * w + 3]));
                            __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 4]), __uint_as_float(r[8 * w + 5]));
                            __nv_bfloat162 p3 = __floats2bfloat162_rn(__uint_as_float(r[8 * w + 6]), __uint_as_float(r[8 * w + 7]));
                            o.x = *reinterpret_cast<uint32_t *>(&p0);
                            o.y = *reinterpret_cast<uint32_t *>(&p1);
                            o.z = *reinterpret_cast<uint32_t *>(&p2);
                            o.w = *reinterpret_cast<uint32_t *>(&p3);
                            dst[w] = o;
                        }
                    }
                }
                ++u;
            } else {
                constexpr int NCH = C::EPI_COLS / 32;
                float acc[C::EPI_COLS];
#pragma unroll
                for (int x = 0; x < C::EPI_COLS; ++x) acc[x] = 0.0f;
                const int MB = (tt.Mg + 31) / 32;
                const int mb = tt.m0 / 32 + q;
                const bool mb_ok = mb < MB;
                const float *sa_row = e.sA + static_cast<int64_t>(mb_ok ? mb : 0) * c.KB;
                const float *sb_row = e.sB + static_cast<int64_t>((tt.n0 + col0) / 32) * c.KB;
                int nb_valid = (c.N - (tt.n0 + col0)) / 32;   // column blocks of this warp inside N
                nb_valid = nb_valid < 0 ? 0 : (nb_valid > NCH ? NCH : nb_valid);
                for (int kb = 0; kb < c.KB; ++kb) {
                    // scale products for this K block (the same for all lanes)
                    const float sa = mb_ok ? __ldg(sa_row + kb) : 0.0f;
                    float sc[NCH];
#pragma unroll
                    for (int x = 0; x < NCH; ++x)
                        sc[x] = (x < nb_valid) ? sa * __ldg(sb_row + static_cast<int64_t>(x) * c.KB + kb) : 0.0f;
                    const uint32_t buf = u & 1u;
                    ok = wait_bar(&ctl->tfull[buf], (u >> 1) & 1u, ctl, c);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t r[NCH][32];
#pragma unroll
                    for (int x = 0; x < NCH; ++x) tmem_ld_x32(tmem + lane_base + buf * BN + col0 + 32 * x, r[x]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                    ++u;
#pragma unroll
                    for (int x = 0; x < NCH; ++x)
#pragma unroll
                        for (int y = 0; y < 32; ++y)
                            acc[32 * x + y] = fmaf(sc[x], __uint_as_float(r[x][y]), acc[32 * x + y]);
                }
                if (!ok) break;
                if (row_ok) {
#pragma unroll
                    for (int x = 0; x < NCH; ++x) {
                        const int col = col0 + 32 * x;
                        if (tt.n0 + col >= c.N) continue;
                        uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint4 o;
                            __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[32 * x + 8 * w + 0], acc[32 * x + 8 * w + 1]);
                            __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[32 * x + 8 * w + 2], acc[32 * x + 8 * w + 3]);
                            __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[32 * x + 8 * w + 4], acc[32 * x + 8 * w + 5]);
                            __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[32 * x + 8 * w + 6], acc[32 * x + 8 * w + 7]);
                            o.x = *reinterpret_cast<uint32_t *>(&p0);
                            o.y = *reinterpret_cast<uint32_t *>(&p1);
                            o.z = *reinterpret_cast<uint32_t *>(&p2);
                            o.w = *reinterpret_cast<uint32_t *>(&p3);
                            dst[w] = o;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->vempty[v]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1) bsfp8_gemm_plain(const __grid_constant__ PlainArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, false>(args, smem_raw);
}

template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1) bsfp8_gemm_grouped(const __grid_constant__ GroupedArgs args) {
    extern __shared__ uint8_t smem_raw[];
    gemm_body<BN, true>(args, smem_raw);
}

// C = 0 for K == 0 (an empty sum).
__global__ void bsfp8_zero_fill(uint4 *p, int64_t n16) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace bsfp8

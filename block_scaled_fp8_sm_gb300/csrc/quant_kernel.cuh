// quant_kernel.cuh -- block quantization of bf16 activations to the GEMM's
// operand format: E4M3 codes with one fp32 scale per 32x32 block, s = amax/448
// (1 for an all-zero block) and q = E4M3(x / s), nearest-even, saturating
// (FP8 GEMM library article, hncyxsy.com/news/241433, sections 2.1-2.2).
//
// HBM-bound: 2 bytes read and 1 byte written per element, plus 4 bytes per
// 1024 elements of scales.  One CTA of 256 threads covers a strip of 32 rows x
// 256 columns (eight blocks): warp w reads rows w, w+8, w+16 and w+24 of the
// strip, lane l the 16 bytes of columns 8l..8l+7, so every warp-row load is
// 512 contiguous bytes and every warp-row store 256.  Block b of the strip is
// held by lanes 4b..4b+3 of all eight warps: its maximum magnitude is taken on
// packed bf16 pairs, reduced over those four lanes with shuffles, then over the
// warps through shared memory.  Five CTAs stay resident per SM (48 registers).
//
// The kernel is bound by its integer/logic pipe rather than by HBM once the
// per-element work is a division, so the arithmetic is kept to a few packed
// instructions per element pair:
//   * s = RN(amax/448) as RN(y + RN(amax - 448 y) / 448) with y = RN(amax r),
//     r = RN(1/448) -- Markstein's correction (P. Markstein, IBM J. Res.
//     Develop. 34(1), 1990) -- equal to the correctly rounded division for
//     every positive finite bf16 amax (checked by enumeration);
//   * x/s from one reciprocal rc = RN(1/s) per block with the same correction,
//     evaluated on -x/s so that no operand needs negating in the packed f32x2
//     form: y' = RN(x (-rc)), e = RN(x + y' s), n = RN(y' + e (-rc)) = -RN(x/s)
//     wherever the residual e is exact; the E4M3 code of -v is the code of v
//     with bit 7 flipped, so the codes are XORed with 0x80.  Enumerating every
//     positive bf16 amax and every bf16 x with |x| <= amax shows that for
//     scales s >= 2^-100 the result equals RN(x/s) wherever |x/s| >= 2^-10 and
//     every code equals that of the correctly rounded division (below 2^-10
//     both codes are +-0).  Smaller or non-finite scales divide (x by -s).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace bsfp8 {

constexpr int QT_COLS = 256;
constexpr int QT_THREADS = 256;
constexpr int QT_MIN_CTAS = 5;   // resident CTAs per SM the register budget is set for

// Two fp32 values -> two E4M3 codes (nearest-even, saturating), lo in byte 0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Running maximum of |x| over packed bf16 pairs (maxNum: a NaN operand is
// ignored, as the oracle's comparison ignores it).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    uint32_t a, d;
    asm("abs.bf16x2 %0, %1;" : "=r"(a) : "r"(w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(acc), "r"(a));
    return d;
}

// s = amax / 448 correctly rounded (1 for an all-zero block; an infinite
// maximum keeps s = inf, as the division gives).
__device__ __forceinline__ float block_scale(float amax) {
    constexpr float kR448 = 0x1.24924ap-9f;   // RN(1/448)
    const float y = __fmul_rn(amax, kR448);
    const float s = __fmaf_rn(__fmaf_rn(-y, 448.0f, amax), kR448, y);
    return amax > 0.0f ? (amax <= 3.40282347e38f ? s : amax) : 1.0f;
}

// The 8 codes of one lane's row segment: word j holds columns 2j (low half)
// and 2j+1 (high half).  RECIP: finite s >= 2^-100 with nrc = -RN(1/s).
template <bool RECIP>
__device__ __forceinline__ uint2 codes8(const uint32_t (&w)[4], float s, float nrc) {
    float v[8];
    if constexpr (RECIP) {
        const uint64_t nr2 = f32x2_pack(__float_as_uint(nrc), __float_as_uint(nrc));
        const uint64_t s2 = f32x2_pack(__float_as_uint(s), __float_as_uint(s));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint64_t x2 = f32x2_pack(w[j] << 16, w[j] & 0xFFFF0000u);
            const uint64_t y2 = mul_f32x2_rn(x2, nr2);    // -y
            const uint64_t e2 = fma_f32x2_rn(y2, s2, x2);  // x - y s
            uint32_t lo, hi;
            f32x2_unpack(fma_f32x2_rn(e2, nr2, y2), lo, hi);   // -(y + e r)
            v[2 * j] = __uint_as_float(lo);
            v[2 * j + 1] = __uint_as_float(hi);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __fdiv_rn(__uint_as_float(w[j] << 16), -s);
            v[2 * j + 1] = __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), -s);
        }
    }
    return make_uint2(__byte_perm(e4m3x2(v[0], v[1]), e4m3x2(v[2], v[3]), 0x5410) ^ 0x80808080u,
                      __byte_perm(e4m3x2(v[4], v[5]), e4m3x2(v[6], v[7]), 0x5410) ^ 0x80808080u);
}

// One 32 x 32 block held by a warp, one row per lane: the lane's 32 bf16 values
// in bf[16] (columns 2j and 2j+1 in word j).  Returns the block's scale (its
// maximum over all 32 lanes) and leaves the lane's 32 codes in codes[8] (byte b
// of word w: column 4w + b) -- the quantizer's arithmetic above, so the codes
// and scale equal those of fp8_quantize_blocks on the same bf16 values.  Every
// lane of the warp must call it (shuffles); rows that do not exist pass zeros.
__device__ __forceinline__ float quantize_rows32(const uint32_t (&bf)[16], uint32_t (&codes)[8]) {
    uint32_t am2 = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) am2 = absmax_bf16x2(am2, bf[j]);
    float amax = fmaxf(__uint_as_float(am2 << 16), __uint_as_float(am2 & 0xFFFF0000u));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float sc = block_scale(amax);
    const bool recip = sc >= 0x1p-100f && sc <= 3.40282347e38f;   // the same for the whole warp
    const float nrc = recip ? -__frcp_rn(sc) : 0.0f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t w[4] = {bf[4 * g], bf[4 * g + 1], bf[4 * g + 2], bf[4 * g + 3]};
        const uint2 cc = recip ? codes8<true>(w, sc, nrc) : codes8<false>(w, sc, 0.0f);
        codes[2 * g] = cc.x;
        codes[2 * g + 1] = cc.y;
    }
    return sc;
}

// Codes of the lane's four rows of the strip (the path is chosen once per strip).
template <bool RECIP>
__device__ __forceinline__ void store_codes(const uint32_t (&w)[4][4], float s, float nrc, uint8_t *q, int64_t r0,
                                            int64_t col, bool col_ok, int64_t M, int64_t K) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + 8 * i;
        const uint2 out = codes8<RECIP>(w[i], s, nrc);
        if (col_ok && r < M) *reinterpret_cast<uint2 *>(q + r * K + col) = out;
    }
}

__global__ void __launch_bounds__(QT_THREADS, QT_MIN_CTAS) bsfp8_quantize_blocks(const __nv_bfloat16 *__restrict__ x,
                                                                                   uint8_t *__restrict__ q,
                                                                                   float *__restrict__ s, int64_t M,
                                                                                   int64_t K) {
    __shared__ float part[QT_THREADS / 32][QT_COLS / 32];   // [warp][block] maxima
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * QT_COLS + 8 * lane;
    const bool col_ok = col < K;   // K is a multiple of 32: 8-column groups are whole
    const int64_t MB = (M + 31) / 32, KB = K / 32;
    for (int64_t mb = blockIdx.y; mb < MB; mb += gridDim.y) {
        const int64_t r0 = mb * 32 + warp;
        uint32_t w[4][4];
        uint32_t am2 = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = r0 + 8 * i;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (col_ok && r < M) raw = *reinterpret_cast<const uint4 *>(x + r * K + col);
            w[i][0] = raw.x;
            w[i][1] = raw.y;
            w[i][2] = raw.z;
            w[i][3] = raw.w;
#pragma unroll
            for (int j = 0; j < 4; ++j) am2 = absmax_bf16x2(am2, w[i][j]);
        }
        float amax = fmaxf(__uint_as_float(am2 << 16), __uint_as_float(am2 & 0xFFFF0000u));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        if ((lane & 3) == 0) part[warp][lane >> 2] = amax;
        __syncthreads();
        float bmax = part[0][lane >> 2];
#pragma unroll
        for (int w8 = 1; w8 < QT_THREADS / 32; ++w8) bmax = fmaxf(bmax, part[w8][lane >> 2]);
        __syncthreads();   // part is rewritten by the next row block
        const float sc = block_scale(bmax);
        if (warp == 0 && (lane & 3) == 0 && col_ok) s[mb * KB + col / 32] = sc;
        if (sc >= 0x1p-100f && sc <= 3.40282347e38f)
            store_codes<true>(w, sc, -__frcp_rn(sc), q, r0, col, col_ok, M, K);
        else
            store_codes<false>(w, sc, 0.0f, q, r0, col, col_ok, M, K);
    }
}

}  // namespace bsfp8

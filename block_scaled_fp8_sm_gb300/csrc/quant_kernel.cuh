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
// held by lanes 4b..4b+3 of all eight warps: its maximum is reduced over those
// four lanes with shuffles, then over the warps through shared memory.
// s is a correctly rounded fp32 division.  The element quotients x/s share one
// reciprocal per block (quotient() below), which takes a third of the issue
// slots of a division per element.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace bsfp8 {

constexpr int QT_COLS = 256;
constexpr int QT_THREADS = 256;

// x/s from r = RN(1/s): y = RN(x r), then Markstein's correction
// q = RN(y + r RN(x - y s)) (P. Markstein, IBM J. Res. Develop. 34(1), 1990,
// the division theorem), which is RN(x/s) whenever the residual x - y s is
// exact.  Used for finite scales s >= 2^-100 only.  Enumerating every positive
// bf16 block maximum (s = RN(amax/448)) and every bf16 x with |x| <= amax
// gives: q == RN(x/s) bit for bit wherever |x/s| >= 2^-10, and below 2^-10
// (subnormal x, underflowing quotients) both lie under half the smallest E4M3
// subnormal, so the code is +-0 either way -- the codes equal those of the
// correctly rounded division for every input.  Below 2^-100, x may be subnormal
// next to quotients that matter, and the kernel divides.
__device__ __forceinline__ float quotient(float x, float s, float r) {
    const float y = __fmul_rn(x, r);
    const float e = __fmaf_rn(-y, s, x);
    const float q = __fmaf_rn(e, r, y);
    return x == 0.0f ? x : q;   // keeps the sign of a zero
}

// Two fp32 values -> two E4M3 codes (nearest-even, saturating), lo in byte 0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(QT_THREADS) bsfp8_quantize_blocks(const __nv_bfloat16 *__restrict__ x,
                                                                      uint8_t *__restrict__ q,
                                                                      float *__restrict__ s, int64_t M,
                                                                      int64_t K) {
    __shared__ float part[QT_THREADS / 32][QT_COLS / 32];   // [warp][block] maxima
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * QT_COLS + 8 * lane;
    const bool col_ok = col < K;   // K is a multiple of 32: 8-column groups are whole
    const int64_t MB = (M + 31) / 32, KB = K / 32;
    for (int64_t mb = blockIdx.y; mb < MB; mb += gridDim.y) {
        float v[4][8];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = mb * 32 + warp + 8 * i;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (col_ok && r < M) raw = *reinterpret_cast<const uint4 *>(x + r * K + col);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[i][2 * j] = __uint_as_float(w[j] << 16);
                v[i][2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                amax = fmaxf(amax, fmaxf(fabsf(v[i][2 * j]), fabsf(v[i][2 * j + 1])));
            }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        if ((lane & 3) == 0) part[warp][lane >> 2] = amax;
        __syncthreads();
        float bmax = part[0][lane >> 2];
#pragma unroll
        for (int w = 1; w < QT_THREADS / 32; ++w) bmax = fmaxf(bmax, part[w][lane >> 2]);
        __syncthreads();   // part is rewritten by the next row block
        const float sc = bmax > 0.0f ? __fdiv_rn(bmax, 448.0f) : 1.0f;
        if (warp == 0 && (lane & 3) == 0 && col_ok) s[mb * KB + col / 32] = sc;
        // The branch is uniform over the lanes of a block, and taken once per
        // 32 elements rather than per element.
        if (sc >= 0x1p-100f && sc <= 3.40282347e38f) {
            const float rc = __frcp_rn(sc);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) v[i][j] = quotient(v[i][j], sc, rc);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) v[i][j] = __fdiv_rn(v[i][j], sc);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = mb * 32 + warp + 8 * i;
            if (!(col_ok && r < M)) continue;
            uint2 out;
            out.x = e4m3x2(v[i][0], v[i][1]) | (e4m3x2(v[i][2], v[i][3]) << 16);
            out.y = e4m3x2(v[i][4], v[i][5]) | (e4m3x2(v[i][6], v[i][7]) << 16);
            *reinterpret_cast<uint2 *>(q + r * K + col) = out;
        }
    }
}

}  // namespace bsfp8

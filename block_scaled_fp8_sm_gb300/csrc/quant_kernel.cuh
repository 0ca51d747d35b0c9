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
// Both divisions are correctly rounded fp32 divisions.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace bsfp8 {

constexpr int QT_COLS = 256;
constexpr int QT_THREADS = 256;

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
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = mb * 32 + warp + 8 * i;
            if (!(col_ok && r < M)) continue;
            uint2 out;
            out.x = e4m3x2(__fdiv_rn(v[i][0], sc), __fdiv_rn(v[i][1], sc)) |
                    (e4m3x2(__fdiv_rn(v[i][2], sc), __fdiv_rn(v[i][3], sc)) << 16);
            out.y = e4m3x2(__fdiv_rn(v[i][4], sc), __fdiv_rn(v[i][5], sc)) |
                    (e4m3x2(__fdiv_rn(v[i][6], sc), __fdiv_rn(v[i][7], sc)) << 16);
            *reinterpret_cast<uint2 *>(q + r * K + col) = out;
        }
    }
}

}  // namespace bsfp8

// tc_common.cuh -- device helpers shared by the TMA + tcgen05 GEMM kernels:
// the grouped tile order and the epilogue's row-chunk store.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace tg {
namespace dev {

// Grouped tile order: tiles are visited in groups of `group_m` tile-rows,
// column by column inside a group.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int& tm, int& tn)
{
    const int span = group_m * tiles_n;
    const int g = t / span;
    const int first = g * group_m;
    const int gs = min(tiles_m - first, group_m);
    const int r = t - g * span;
    tm = first + r % gs;
    tn = r / gs;
}

// Stores 32 consecutive fp32 accumulator values r[0..31] of row m, columns
// n..n+31, converted to the output type; columns >= N are skipped.
template <bool OUT_F32>
__device__ __forceinline__ void store_chunk(void* C, long long ldc, int m, int n, int N,
                                            const uint32_t* r, bool vec)
{
    if constexpr (OUT_F32) {
        float* row = static_cast<float*>(C) + static_cast<long long>(m) * ldc + n;
        if (vec && n + 32 <= N) {
            float4* d = reinterpret_cast<float4*>(row);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                d[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n + j < N) row[j] = __uint_as_float(r[j]);
        }
    } else {
        __half* row = static_cast<__half*>(C) + static_cast<long long>(m) * ldc + n;
        if (vec && n + 32 <= N) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                __half2 h = __floats2half2_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                p[i] = *reinterpret_cast<uint32_t*>(&h);
            }
            uint4* d = reinterpret_cast<uint4*>(row);
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n + j < N) row[j] = __float2half_rn(__uint_as_float(r[j]));
        }
    }
}

}  // namespace dev
}  // namespace tg

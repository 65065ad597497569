// tc_common.cuh -- device helpers shared by the GEMM kernels: the grouped
// tile order, the fused epilogue and the epilogue's row-chunk store.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tg_internal.h"

namespace tg {
namespace dev {

// Grouped tile order: tiles are visited in groups of `group_m` tile-rows,
// column by column inside a group, left to right in even groups and right to
// left in odd ones, so a group starts on the B columns its predecessor read
// last.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int& tm, int& tn)
{
    const int span = group_m * tiles_n;
    const int g = t / span;
    const int first = g * group_m;
    const int gs = min(tiles_m - first, group_m);
    const int r = t - g * span;
    tm = first + r % gs;
    tn = (g & 1) ? tiles_n - 1 - r / gs : r / gs;
}

// Tile t of a strided batch of matrices, each tiles_m x tiles_n tiles walked
// in the grouped order: b is the matrix, (tm, tn) the tile inside it.
__device__ __forceinline__ void batch_tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                                  int& b, int& tm, int& tn)
{
    const int per = tiles_m * tiles_n;
    b = t / per;
    tile_coords(t - b * per, tiles_m, tiles_n, group_m, tm, tn);
}

// Matrix b of a strided batch of C (stride sC elements of es bytes).
__device__ __forceinline__ void* batch_ptr(void* C, int b, long long sC, int es)
{
    return static_cast<char*>(C) + static_cast<long long>(b) * sC * es;
}

// GELU is x * Phi(x) with Phi the standard normal distribution function,
// written as 0.5 * x * erfc(-x / sqrt(2)) so the negative tail keeps its
// relative accuracy.  Kept out of line: the epilogue applies it to 32
// unrolled values, and 32 inlined copies of erfc double the pair kernel's
// registers and, measured with eight epilogue warps, run no faster.
static __device__ __noinline__ float gelu(float y)
{
    return 0.5f * y * erfcf(-0.70710678118654752f * y);
}

// Activation of the fused epilogue.  fmaxf maps NaN to 0, as "x > 0 ? x : 0"
// does.
__device__ __forceinline__ float act_apply(float y, int act)
{
    if (act == ACT_RELU) return fmaxf(y, 0.0f);
    if (act == ACT_GELU) return gelu(y);
    return y;
}

// One output element of the fused epilogue: act(alpha*acc + bias[n] + beta*D[m,n]).
template <bool OUT_F32>
__device__ __forceinline__ float epilogue_elem(float acc, int m, int n, const Epilogue& e)
{
    float y = e.alpha * acc;
    if (e.bias) y += __ldg(e.bias + n);
    if (e.beta != 0.0f) {
        const long long i = static_cast<long long>(m) * e.ldd + n;
        const float d = OUT_F32 ? static_cast<const float*>(e.D)[i]
                                : __half2float(static_cast<const __half*>(e.D)[i]);
        y = fmaf(e.beta, d, y);
    }
    return act_apply(y, e.act);
}

// The fused epilogue over 32 accumulators r[0..31] (fp32 bit patterns) of row
// m, columns n..n+31, in place; columns >= N are left as they are (the store
// skips them).  D is read with plain loads, never through the read-only
// path, because it may be C itself.
template <bool OUT_F32>
__device__ __forceinline__ void epilogue_chunk(uint32_t* r, int m, int n, int N, const Epilogue& e)
{
    const bool full = n + 32 <= N;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = e.alpha * __uint_as_float(r[j]);
    if (e.bias) {
        if (e.bias_vec && full) {
            const float4* b = reinterpret_cast<const float4*>(e.bias + n);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = __ldg(b + i);
                v[4 * i] += q.x;
                v[4 * i + 1] += q.y;
                v[4 * i + 2] += q.z;
                v[4 * i + 3] += q.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n + j < N) v[j] += __ldg(e.bias + n + j);
        }
    }
    if (e.beta != 0.0f) {
        const long long row = static_cast<long long>(m) * e.ldd + n;
        if constexpr (OUT_F32) {
            const float* d = static_cast<const float*>(e.D) + row;
            if (e.d_vec && full) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 q = reinterpret_cast<const float4*>(d)[i];
                    v[4 * i] = fmaf(e.beta, q.x, v[4 * i]);
                    v[4 * i + 1] = fmaf(e.beta, q.y, v[4 * i + 1]);
                    v[4 * i + 2] = fmaf(e.beta, q.z, v[4 * i + 2]);
                    v[4 * i + 3] = fmaf(e.beta, q.w, v[4 * i + 3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (n + j < N) v[j] = fmaf(e.beta, d[j], v[j]);
            }
        } else {
            const __half* d = static_cast<const __half*>(e.D) + row;
            if (e.d_vec && full) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 q = reinterpret_cast<const uint4*>(d)[i];
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                        v[8 * i + 2 * k] = fmaf(e.beta, f.x, v[8 * i + 2 * k]);
                        v[8 * i + 2 * k + 1] = fmaf(e.beta, f.y, v[8 * i + 2 * k + 1]);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (n + j < N) v[j] = fmaf(e.beta, __half2float(d[j]), v[j]);
            }
        }
    }
    if (e.act != ACT_NONE) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = act_apply(v[j], e.act);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
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

// One epilogue warp's 32 x 32 chunk of C (rows m0..m0+31, lane = row,
// columns n..n+31, r[] the lane's fp32 accumulators after the fused
// epilogue) through shared memory and one TMA store: the lane writes its
// row, converted, into the warp's staging buffer `slot` (64 B per row for
// fp16, 128 B for fp32), and lane 0 stores the box [32 cols][32 rows] at
// (n, m0, z) of `tmC`; the TMA engine writes only the part inside C.  The
// warp's 32 rows then leave as one bulk copy instead of 32-row scattered
// 16-byte stores.  The caller keeps `slot` untouched until the store has
// read it (bulk_wait_read in lane 0, then __syncwarp).
template <bool OUT_F32>
__device__ __forceinline__ void stage_store_chunk(const CUtensorMap* tmC, uint32_t slot,
                                                  const uint32_t* r, int n, int m0, int z,
                                                  int lane)
{
    if constexpr (OUT_F32) {
        const uint32_t row = slot + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            st_shared_v4(row + 16u * i, r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
    } else {
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __half2 h = __floats2half2_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            p[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        const uint32_t row = slot + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
        for (int i = 0; i < 4; ++i) st_shared_v4(row + 16u * i, p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
    }
    fence_proxy_async_smem();  // the rows are visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmC, slot, n, m0, z);
        bulk_commit();
    }
}

// One epilogue warp's 32-row x 128-byte box of C through shared memory and
// one TMA store: rows m0..m0+31 (lane = row), 64 fp16 or 32 fp32 columns
// from n, r[] the lane's fp32 accumulators after the fused epilogue (64 for
// fp16 output, 32 for fp32).  The lane writes its row, converted, into the
// warp's 4 KB staging buffer `slot` (128 bytes per row), and lane 0 stores
// the box at (n, m0, z) of `tmC`; the TMA engine writes only the part
// inside C.  The warp's rows then leave as one bulk copy instead of 32
// scattered 16-byte stores per instruction.  The caller keeps `slot`
// untouched until the store has read it (bulk_wait_read in lane 0, then
// __syncwarp).
template <bool OUT_F32>
__device__ __forceinline__ void stage_store_box(const CUtensorMap* tmC, uint32_t slot,
                                                const uint32_t* r, int n, int m0, int z,
                                                int lane)
{
    const uint32_t row = slot + static_cast<uint32_t>(lane) * 128u;
    if constexpr (OUT_F32) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            st_shared_v4(row + 16u * i, r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 h = __floats2half2_rn(__uint_as_float(r[8 * i + 2 * j]),
                                              __uint_as_float(r[8 * i + 2 * j + 1]));
                p[j] = *reinterpret_cast<uint32_t*>(&h);
            }
            st_shared_v4(row + 16u * i, p[0], p[1], p[2], p[3]);
        }
    }
    fence_proxy_async_smem();  // the rows are visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmC, slot, n, m0, z);
        bulk_commit();
    }
}

}  // namespace dev
}  // namespace tg

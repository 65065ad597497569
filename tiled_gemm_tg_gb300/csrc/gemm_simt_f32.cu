// gemm_simt_f32.cu -- fp32 GEMM on the CUDA cores (fp32 in, fp32 accumulate,
// fp32 out), and the elementwise kernel of a fused epilogue over an empty
// product (K == 0).
//
// This serves the fp32 128x128x128 example of "TileLang实战：用Python DSL自动
// 生成高性能GPU计算内核" (gsyq.cn), §3.1 (the triple loop C[i,j] += A[i,k] *
// B[k,j]) and §3.2 (checked against NumPy within 1e-4), with the shared-
// memory tiling idea of that page's §5.3 restated correctly: each CTA stages
// an A tile and the matching B tile (the page's snippet indexes B with A's
// coordinates, which is not a matrix product).
//
// Tiling: a CTA computes a 64 x 64 tile of C with 256 threads; each thread
// owns a 4 x 4 register block and accumulates it with fmaf in ascending k.
// A is staged transposed ([BK][BM]) so a thread reads its four A values as
// one float4; both tiles are double-buffered so the loads of k-block i+1
// overlap the FMAs of k-block i.  Every global access is predicated, so any
// M, N, K and row strides work.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

using namespace tg::dev;

constexpr int BM = 64;
constexpr int BN = 64;
constexpr int BK = 16;
constexpr int TM = 4;
constexpr int TN = 4;
constexpr int kThreads = (BM / TM) * (BN / TN);  // 256

__global__ void __launch_bounds__(kThreads)
gemm_simt_f32_kernel(const float* __restrict__ A0, long long lda, const float* __restrict__ B0,
                     long long ldb, float* C0, long long ldc, int M, int N, int K, Epilogue epi,
                     BatchArgs bt)
{
    // grid.z walks the matrices of a strided batch
    const long long bz = blockIdx.z;
    const float* const A = A0 + bz * bt.sA;
    const float* const B = B0 + bz * bt.sB;
    float* const C = C0 + bz * bt.sC;
    __shared__ __align__(16) float As[2][BK][BM + 4];  // +4: fewer bank conflicts on the transposing store
    __shared__ __align__(16) float Bs[2][BK][BN];

    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN);  // column block
    const int ty = tid / (BN / TN);  // row block
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * BN;

    // Each thread moves 4 A elements and 4 B elements per k-block.
    float ra[4], rb[4];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + i * kThreads;       // 0 .. 1023
            const int am = e / BK, ak = e % BK;     // A tile: 64 rows x 16 k
            const int gm = m0 + am, gk = k0 + ak;
            ra[i] = (gm < M && gk < K) ? __ldg(A + static_cast<long long>(gm) * lda + gk) : 0.0f;
            const int bk = e / BN, bn = e % BN;     // B tile: 16 k x 64 cols
            const int hk = k0 + bk, hn = n0 + bn;
            rb[i] = (hk < K && hn < N) ? __ldg(B + static_cast<long long>(hk) * ldb + hn) : 0.0f;
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + i * kThreads;
            As[buf][e % BK][e / BK] = ra[i];
            Bs[buf][e / BN][e % BN] = rb[i];
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    const int num_kb = (K + BK - 1) / BK;
    fetch(0);
    stash(0);
    __syncthreads();
    for (int kb = 0; kb < num_kb; ++kb) {
        const int buf = kb & 1;
        if (kb + 1 < num_kb) fetch((kb + 1) * BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * TM]);
            const float4 b4 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * TN]);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w};
            const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kb + 1 < num_kb) stash(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = m0 + ty * TM + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + tx * TN + j;
            if (n < N)
                C[static_cast<long long>(m) * ldc + n] =
                    epi.on ? epilogue_elem<true>(acc[i][j], m, n, epi) : acc[i][j];
        }
    }
}

// K == 0: the product is the empty sum, so each element is act(beta * D +
// bias), or 0 without an epilogue.  One thread per column, rows strided over
// grid.y, the matrices of a strided batch over grid.z.
template <bool OUT_F32>
__global__ void __launch_bounds__(256)
epilogue_only_kernel(void* C0, long long ldc, int M, int N, Epilogue epi, long long sC)
{
    const int n = blockIdx.x * 256 + static_cast<int>(threadIdx.x);
    if (n >= N) return;
    void* const C = batch_ptr(C0, static_cast<int>(blockIdx.z), sC, OUT_F32 ? 4 : 2);
    for (int m = blockIdx.y; m < M; m += gridDim.y) {
        const float y = epi.on ? epilogue_elem<OUT_F32>(0.0f, m, n, epi) : 0.0f;
        const long long i = static_cast<long long>(m) * ldc + n;
        if constexpr (OUT_F32)
            static_cast<float*>(C)[i] = y;
        else
            static_cast<__half*>(C)[i] = __float2half_rn(y);
    }
}

}  // namespace

cudaError_t launch_epilogue_only(const GemmArgs& a)
{
    const unsigned gx = static_cast<unsigned>((static_cast<long long>(a.N) + 255) / 256);
    const unsigned gy = static_cast<unsigned>(a.M < 65535 ? a.M : 65535);
    if (a.batch > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid(gx, gy, a.batch);
    if (a.out_f32)
        epilogue_only_kernel<true><<<grid, 256, 0, a.stream>>>(a.C, a.ldc, a.M, a.N, a.epi, a.sC);
    else
        epilogue_only_kernel<false><<<grid, 256, 0, a.stream>>>(a.C, a.ldc, a.M, a.N, a.epi, a.sC);
    return cudaGetLastError();
}

cudaError_t launch_simt_f32(const GemmArgs& a)
{
    const dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, a.batch);
    if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
    gemm_simt_f32_kernel<<<grid, kThreads, 0, a.stream>>>(
        static_cast<const float*>(a.A), a.lda, static_cast<const float*>(a.B), a.ldb,
        static_cast<float*>(a.C), a.ldc, a.M, a.N, a.K, a.epi, a.batch_args());
    return cudaGetLastError();
}

}  // namespace tg

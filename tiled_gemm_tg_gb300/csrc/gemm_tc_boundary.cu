// gemm_tc_boundary.cu -- fp16 GEMM on the tensor cores for operands the TMA
// engine cannot address: a base pointer that is not 16-byte aligned or a row
// stride that is not a multiple of 16 bytes (e.g. B of the M=127, N=255 case
// has a 510-byte row stride; a 4x4 fp16 matrix has an 8-byte one).
//
// The pages require such unaligned shapes to work without reading out of
// bounds or writing garbage (gsyq.cn/news/429607, §3.3 第三步 and §5.2); the
// tile masking is what they call for.  Here every global load is predicated
// and zero-filled, written by the threads themselves into the same 128-byte
// swizzled shared-memory layout the TMA path produces, and fed to the same
// tcgen05.mma (M=128, N=BN, K=16) with an fp32 accumulator in tensor memory.
// Each thread issues all its loads of k-block i+1 into registers while the
// tensor core runs k-block i; two shared-memory stages.  4 warps; stores
// predicated.
//
// Loads that cannot be 16 bytes wide are latency-bound, so a problem with few
// 128 x BN output tiles is also split over K: a cluster of S CTAs (S = 2, 4
// or 8) shares one output tile, CTA r taking k-blocks [r*nkb/S, (r+1)*nkb/S).
// Each CTA writes its fp32 partial tile into its own shared memory (rows
// padded by four floats, so the writes from tensor-memory lanes do not
// collide on banks), the cluster synchronises, and CTA r adds up, in rank
// order, rows [r*128/S, (r+1)*128/S) of all S partials through distributed
// shared memory, applies the epilogue and stores them.  With S = 1 (enough
// tiles to fill the GPU) each CTA stores its tile straight from tensor
// memory.
#include <cstdint>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

using namespace tg::dev;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;
constexpr uint32_t A_STAGE = BM * BK * 2;   // 16 KB
constexpr uint32_t B_STAGE = BN * BK * 2;   // 16 KB: two [64 k][64 n] atoms-columns
constexpr uint32_t STAGE = A_STAGE + B_STAGE;
constexpr int RED_LD = BN + 4;                       // floats per partial row
constexpr uint32_t RED_BYTES = BM * RED_LD * 4;      // fp32 partial tile, 66 KB
constexpr uint32_t SMEM = (2 * STAGE > RED_BYTES ? 2 * STAGE : RED_BYTES) + 1024;
constexpr int kMaxSplit = 8;
constexpr uint32_t TMEM_COLS = BN;
constexpr int kThreads = 128;

// One k-block of operands held in registers: each thread's 8 chunks of the
// A tile (128 rows x 8 chunks of 8 k) and 8 chunks of the B tile (64 k-rows x
// BN/8 chunks of 8 n).  A chunk is either one 16-byte load (operand 16-byte
// aligned, chunk in range) or eight 2-byte loads, each in its own register.
// Every load of the k-block is issued before any value is used: the GPU
// issues in order, so packing a value right after its load would stall the
// thread before the next chunk's loads went out.
constexpr int kChunksA = BM * (BK / 8) / kThreads;
constexpr int kChunksB = BK * (BN / 8) / kThreads;
static_assert(kChunksA * kThreads == BM * (BK / 8) && kChunksB * kThreads == BK * (BN / 8),
              "tile chunks must divide evenly over the threads");

struct Frag {
    uint32_t a[kChunksA][8];
    uint32_t b[kChunksB][8];
    uint32_t wide;  // bit j: A chunk j was one 16-byte load; bit 8 + j: B chunk j
};

__device__ __forceinline__ void load_chunk(const __half* p, int valid, bool vec, uint32_t (&e)[8],
                                           uint32_t& wide, uint32_t bit)
{
    if (vec && valid >= 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        e[0] = v.x;
        e[1] = v.y;
        e[2] = v.z;
        e[3] = v.w;
        wide |= bit;
    } else {
        const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = (i < valid) ? static_cast<uint32_t>(__ldg(q + i)) : 0u;
    }
}

__device__ __forceinline__ uint4 pack_chunk(const uint32_t (&e)[8], bool wide)
{
    if (wide) return make_uint4(e[0], e[1], e[2], e[3]);
    return make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16),
                      e[6] | (e[7] << 16));
}

__device__ __forceinline__ void fetch(Frag& f, const __half* __restrict__ A, long long lda,
                                      bool a_vec, const __half* __restrict__ B, long long ldb,
                                      bool b_vec, int M, int N, int K, int m0, int n0, int k0,
                                      int tid)
{
    f.wide = 0;
#pragma unroll
    for (int j = 0; j < kChunksA; ++j) {
        const int i = tid + j * kThreads;
        const int r = i >> 3, c = i & 7;
        const int m = m0 + r, k = k0 + c * 8;
        if (m < M && k < K) {
            load_chunk(A + static_cast<long long>(m) * lda + k, K - k, a_vec, f.a[j], f.wide,
                       1u << j);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f.a[j][e] = 0;
        }
    }
#pragma unroll
    for (int j = 0; j < kChunksB; ++j) {
        const int i = tid + j * kThreads;
        const int kr = i / (BN / 8), c = i % (BN / 8);
        const int k = k0 + kr, n = n0 + c * 8;
        if (k < K && n < N) {
            load_chunk(B + static_cast<long long>(k) * ldb + n, N - n, b_vec, f.b[j], f.wide,
                       1u << (8 + j));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f.b[j][e] = 0;
        }
    }
}

// Registers -> one stage, in the 128-byte swizzled layouts the TMA path
// produces: A chunk (r, c) at row r, 16-byte slot c ^ (r % 8); B chunk
// (kr, c) in 64-column box c / 8 (8 KB apart), row kr, slot (c % 8) ^ (kr % 8).
__device__ __forceinline__ void stash(const Frag& f, uint8_t* sA, uint8_t* sB, int tid)
{
#pragma unroll
    for (int j = 0; j < kChunksA; ++j) {
        const int i = tid + j * kThreads;
        const int r = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(sA + r * 128 + ((c ^ (r & 7)) << 4)) =
            pack_chunk(f.a[j], (f.wide >> j) & 1u);
    }
#pragma unroll
    for (int j = 0; j < kChunksB; ++j) {
        const int i = tid + j * kThreads;
        const int kr = i / (BN / 8), c = i % (BN / 8);
        *reinterpret_cast<uint4*>(sB + (c >> 3) * (64 * 128) + kr * 128 +
                                  (((c & 7) ^ (kr & 7)) << 4)) =
            pack_chunk(f.b[j], (f.wide >> (8 + j)) & 1u);
    }
}

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads)
gemm_tc_boundary_kernel(const __half* __restrict__ A0, long long lda, const __half* __restrict__ B0,
                        long long ldb, void* C0, long long ldc, int M, int N, int K, int split,
                        int hook, unsigned int* err, Epilogue epi, BatchArgs bt)
{
    // grid.z walks the matrices of a strided batch
    const int bz = static_cast<int>(blockIdx.z);
    const __half* const A = A0 + static_cast<long long>(bz) * bt.sA;
    const __half* const B = B0 + static_cast<long long>(bz) * bt.sB;
    void* const C = batch_ptr(C0, bz, bt.sC, OUT_F32 ? 4 : 2);
    // An operand whose base and row stride are both 16-byte multiples is read
    // with 16-byte loads (at most one of A and B is, or the TMA path serves).
    const bool a_vec = (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && (lda & 7) == 0;
    const bool b_vec = (reinterpret_cast<uintptr_t>(B) & 15u) == 0 && (ldb & 7) == 0;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int m0 = blockIdx.y * BM;
    // a cluster of `split` CTAs along x shares one output tile
    const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int n0 = static_cast<int>(blockIdx.x / split) * BN;

    if (tid == 0) {
        mbar_init(smem_u32(&mma_bar[0]), 1);
        mbar_init(smem_u32(&mma_bar[1]), 1);
        mbar_init(smem_u32(&drain_bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    pdl_wait();  // the previous kernel on the stream is complete from here on

    constexpr uint32_t idesc = idesc_f16_f32(BM, BN, false, true);
    const int nkb_all = (K + BK - 1) / BK;
    const int kb0 = static_cast<int>(static_cast<long long>(rank) * nkb_all / split);
    const int num_kb = static_cast<int>(static_cast<long long>(rank + 1) * nkb_all / split) - kb0;
    bool aborted = false;

    // Registers carry k-block i+1 while the tensor core works on k-block i
    // (i counts this CTA's k-blocks; kb0 + i is the k-block of the problem).
    Frag f;
    if (num_kb > 0) fetch(f, A, lda, a_vec, B, ldb, b_vec, M, N, K, m0, n0, kb0 * BK, tid);
    for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb & 1;
        if (kb >= 2) {
            // The MMAs issued two k-blocks ago read stage s; wait until done.
            const bool got = mbar_wait(smem_u32(&mma_bar[s]), ((kb - 2) >> 1) & 1, nullptr);
            if (__syncthreads_or(got ? 0 : 1)) {
                aborted = true;
                break;
            }
        }
        uint8_t* sA = gbase + s * STAGE;
        stash(f, sA, sA + A_STAGE, tid);
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sa = base + s * STAGE;
            const uint64_t ad = sdesc_sw128(sa, 16, 1024);
            const uint64_t bd = sdesc_sw128(sa + A_STAGE, BK * 128, 1024);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
                umma_f16(tmem_base, ad + 2ull * k, bd + 128ull * k, idesc, (kb | k) != 0 ? 1u : 0u);
            // test hook: skip the first commit, so the bounded wait on it runs out
            if (!(hook == 1 && kb == 0)) umma_commit(smem_u32(&mma_bar[s]));
        }
        if (kb + 1 < num_kb)
            fetch(f, A, lda, a_vec, B, ldb, b_vec, M, N, K, m0, n0, (kb0 + kb + 1) * BK, tid);
    }

    if (!aborted && num_kb > 0) {
        const int last = num_kb - 1;
        const bool got = mbar_wait(smem_u32(&mma_bar[last & 1]), (last >> 1) & 1, nullptr);
        if (__syncthreads_or(got ? 0 : 1)) aborted = true;
    }
    if (split > 1) {
        // This CTA's partial tile -> its shared memory (the stages are free:
        // every MMA reading them has completed), row m_local at
        // red[m_local * RED_LD]; a CTA without k-blocks contributes zeros.
        float* const red = reinterpret_cast<float*>(gbase);
        if (!aborted) {
            tc_fence_after();
            const int ml = warp * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                if (num_kb > 0) {
                    tmem_ld_32x32b_x32(taddr + c, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                float4* row = reinterpret_cast<float4*>(red + ml * RED_LD + c);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    row[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
        } else if (tid == 0) {
            atomicOr(err, ERR_BOUNDARY);
        }
        // every partial of the cluster is in shared memory after this barrier
        cluster_sync();
        const int span = BM / split;
        const uint32_t red_local = smem_u32(red);
        for (int idx = tid; idx < span * (BN / 4); idx += kThreads) {
            const int ml = rank * span + idx / (BN / 4);
            const int nl = 4 * (idx % (BN / 4));
            const int m = m0 + ml, n = n0 + nl;
            if (m >= M || n >= N) continue;
            const uint32_t off = static_cast<uint32_t>((ml * RED_LD + nl) * 4);
            float4 part[kMaxSplit];
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r)
                if (r < split) {
                    const uint32_t ra = mapa_shared(red_local + off, static_cast<uint32_t>(r));
                    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(part[r].x), "=f"(part[r].y), "=f"(part[r].z), "=f"(part[r].w)
                                 : "r"(ra)
                                 : "memory");
                }
            float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r)
                if (r < split) {
                    sum[0] += part[r].x;
                    sum[1] += part[r].y;
                    sum[2] += part[r].z;
                    sum[3] += part[r].w;
                }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (n + j >= N) break;
                float y = sum[j];
                if (epi.on) y = epilogue_elem<OUT_F32>(y, m, n + j, epi);
                if constexpr (OUT_F32)
                    static_cast<float*>(C)[static_cast<long long>(m) * ldc + n + j] = y;
                else
                    static_cast<__half*>(C)[static_cast<long long>(m) * ldc + n + j] =
                        __float2half_rn(y);
            }
        }
    } else if (!aborted) {
        tc_fence_after();
        const int m = m0 + warp * 32 + lane;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c, r);
            tmem_ld_wait();
            const int n = n0 + c;
            if (m < M && n < N) {
                if (epi.on) epilogue_chunk<OUT_F32>(r, m, n, N, epi);
                if constexpr (OUT_F32) {
                    float* row = static_cast<float*>(C) + static_cast<long long>(m) * ldc + n;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n + j < N) row[j] = __uint_as_float(r[j]);
                } else {
                    __half* row = static_cast<__half*>(C) + static_cast<long long>(m) * ldc + n;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n + j < N) row[j] = __float2half_rn(__uint_as_float(r[j]));
                }
            }
        }
    } else if (tid == 0) {
        atomicOr(err, ERR_BOUNDARY);
    }

    if (tid == 0) {
        // Every MMA this CTA issued must finish before TMEM is freed.
        umma_commit(smem_u32(&drain_bar));
        if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
    }
    pdl_trigger();  // this CTA has issued all its global writes
    // no CTA may leave while a peer can still read its shared memory
    if (split > 1) cluster_sync();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

std::mutex g_attr_mu;
bool g_attr_set[64][2];
// Clusters of 2, 4 and 8 CTAs that can be resident at once, per device and
// output type.
int g_max_clusters[64][2][3];

}  // namespace

int boundary_split(long long tiles, int nkb, int num_sms, const int* max_clusters)
{
    int s = 1;
    for (int i = 0; i < 3; ++i) {
        const int t = 2 << i;
        if (t > kMaxSplit || tiles * t > num_sms || nkb < t ||
            (max_clusters != nullptr && tiles > max_clusters[i]))
            break;
        s = t;
    }
    return s;
}

namespace {

template <bool OUT_F32>
cudaError_t launch_cfg(const GemmArgs& a)
{
    auto kernel = gemm_tc_boundary_kernel<OUT_F32>;
    const int o = OUT_F32 ? 1 : 0;
    int split = 1;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(g_attr_mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!g_attr_set[dev][o]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(SMEM));
            if (e != cudaSuccess) return e;
            for (int i = 0; i < 3; ++i) {
                cudaLaunchConfig_t q = {};
                q.gridDim = dim3(2 << i, 1);
                q.blockDim = dim3(kThreads);
                q.dynamicSmemBytes = SMEM;
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeClusterDimension;
                at[0].val.clusterDim.x = 2 << i;
                at[0].val.clusterDim.y = 1;
                at[0].val.clusterDim.z = 1;
                q.attrs = at;
                q.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, kernel, &q) != cudaSuccess) {
                    cudaGetLastError();
                    n = 0;
                }
                g_max_clusters[dev][o][i] = n;
            }
            g_attr_set[dev][o] = true;
        }
        const long long tiles = static_cast<long long>((a.N + BN - 1) / BN) *
                                ((a.M + BM - 1) / BM) * a.batch;
        split = boundary_split(tiles, (a.K + BK - 1) / BK, a.num_sms, g_max_clusters[dev][o]);
    }
    const long long gx = static_cast<long long>((a.N + BN - 1) / BN) * split;
    if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(gx), (a.M + BM - 1) / BM, a.batch);
    if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = a.stream;
    cudaLaunchAttribute at[2];
    set_pdl_attr(at[0]);
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = split;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = split > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<const __half*>(a.A), a.lda,
                              static_cast<const __half*>(a.B), a.ldb, a.C, a.ldc, a.M, a.N, a.K,
                              split, a.hook, a.err, a.epi, a.batch_args());
}

}  // namespace

cudaError_t launch_boundary(const GemmArgs& a)
{
    return a.out_f32 ? launch_cfg<true>(a) : launch_cfg<false>(a);
}

}  // namespace tg

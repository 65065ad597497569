// gemm_skinny.cu -- fp16 GEMM for small M (M <= 64), the decode-like shapes
// where C = A x B is bound by streaming B from HBM, not by the tensor cores
// (16 x 4096 x 4096: 15.9 FLOP per byte).
//
// It computes the same product as the pages' tiled GEMM ("企业官网建设流程全
// 解析" (cf-1.com) §3.3; "TileLang实战" (gsyq.cn) §3.1), arranged so that B
// streams through every SM:
//   * operands swapped: C^T[N, M] = B^T[N, K] x A^T[K, M].  The MMA's M = 128
//     runs over N (B^T is MN-major in shared memory: B's rows are contiguous
//     in n), the MMA's N = Mp (M rounded up to 16) runs over M (A is K-major);
//     the accumulator holds 128 n-lanes x Mp fp32 columns in TMEM;
//   * split-K over a thread-block cluster of S CTAs (S = 1, 2, 4 or 8, the
//     largest that keeps every cluster of the grid co-resident): CTA r
//     of the cluster owns the same 128 columns of C and k-blocks
//     [r*nkb/S, (r+1)*nkb/S), so n_tiles * S CTAs stream disjoint parts of B;
//   * the S fp32 partials meet in distributed shared memory: each CTA writes
//     its partial (read from TMEM) into its own shared memory, the cluster
//     synchronises, and CTA r sums, in rank order, rows n in
//     [r*128/S, (r+1)*128/S) of all S partials, rounds to the output type and
//     stores them.  No global workspace, one launch.
// Roles (192 threads per CTA): warp 0 TMA producer (k-block 128, four
// stages; a stage's two B^T column blocks, and its two A k-blocks of 64, in
// one 4-D copy each when N, and K, are whole numbers of blocks), warp 1
// TMEM allocation + single-thread tcgen05.mma issue, warps 2-5 read the
// accumulator, one per TMEM lane quadrant.  Waits are bounded; on expiry the kernel records
// a bit in the device error word, stops issuing, waits for its own copies and
// MMAs, and still reaches the cluster barriers so no CTA waits on a missing
// peer.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "l2_prefetch.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

using namespace tg::dev;

constexpr int BNT = 128;                       // n per CTA (the MMA's M)
constexpr int BK = 128;                        // k-block: eight MMAs per stage
constexpr uint32_t BT_BOX = 64 * BK * 2;       // [BK k][64 n] box of B^T, 16 KB
constexpr uint32_t BT_STAGE = BNT * BK * 2;    // 32 KB
constexpr int STAGES = 4;
constexpr int kThreads = 192;
constexpr int kMaxSplit = 8;

template <int MP>
struct SkinnyCfg {
    static constexpr uint32_t A_ATOM = MP * 128;          // [MP rows][64 k]
    static constexpr uint32_t A_STAGE = MP * BK * 2;
    static constexpr uint32_t STAGE = BT_STAGE + A_STAGE;
    static constexpr uint32_t SMEM = STAGES * STAGE + 1024;
    static constexpr uint32_t TMEM_COLS = MP <= 32 ? 32 : 64;
    static constexpr uint32_t RED_BYTES = MP * BNT * 4;  // fp32 partial [MP][128]
    static_assert(SMEM <= 227 * 1024, "shared-memory budget exceeded");
    static_assert(RED_BYTES <= STAGES * STAGE, "reduction buffer must fit in the stages");
};

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t cluster_addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

template <int MP, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBT,
                   void* C, long long ldc, int M, int N, int K, int split, int chunked,
                   int hook, unsigned int* err, Epilogue epi, BatchArgs bt)
{
    using Cfg = SkinnyCfg<MP>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    float* const red = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());  // == blockIdx.x (cluster spans x)
    const int n0 = blockIdx.y * BNT;
    const int bz = static_cast<int>(blockIdx.z);  // matrix of the batch
    void* const Cb = batch_ptr(C, bz, bt.sC, OUT_F32 ? 4 : 2);
    const int nkb = (K + BK - 1) / BK;
    const int kb0 = static_cast<int>(static_cast<long long>(rank) * nkb / split);
    const int kb1 = static_cast<int>(static_cast<long long>(rank + 1) * nkb / split);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&tfull_bar), 1);
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmBT);
        // this CTA's first stages into L2 while the previous kernel finishes
        for (int kb = kb0; kb < kb1 && kb < kb0 + min(STAGES, kPrefetchStagesSingle); ++kb) {
            if (chunked & 1) {
                tma_prefetch_l2_4d(&tmBT, 0, kb * BK, n0 / 64, bz * bt.zb);
            } else {
                for (int j = 0; j < BNT / 64; ++j)
                    tma_prefetch_l2_3d(&tmBT, n0 + j * 64, kb * BK, bz * bt.zb);
            }
            if (chunked & 2) {
                tma_prefetch_l2_4d(&tmA, 0, 0, kb * (BK / 64), bz * bt.za);
            } else {
                for (int j = 0; j < BK / 64; ++j)
                    tma_prefetch_l2_3d(&tmA, kb * BK + j * 64, 0, bz * bt.za);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    pdl_wait();  // the previous kernel on the stream is complete from here on
    const uint32_t epi_limit = kSlowPolls + 64u * static_cast<uint32_t>(min(kb1 - kb0, 1 << 20));

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, &abort_flag)) {
                    abort_flag = 1;
                    atomicOr(err, ERR_SKINNY);
                    break;
                }
                if (hook == 1 && kb == kb0) {
                    // test hook: leave this stage unfilled, so the MMA
                    // thread's bounded wait on it runs out
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    continue;
                }
                const uint32_t fb = smem_u32(&full_bar[s]);
                const uint32_t sa = base + s * Cfg::STAGE;
                mbar_arrive_expect_tx(fb, Cfg::STAGE);
// the stage's column blocks of B^T (and k-blocks of A) in one copy
                // each when the sizes are whole blocks (chunked bit 0 / 1)
                if (chunked & 1) {
                    tma_load_4d(sa, &tmBT, fb, 0, kb * BK, n0 / 64, bz * bt.zb);
                } else {
#pragma unroll
                    for (int j = 0; j < BNT / 64; ++j)
                        tma_load_3d(sa + j * BT_BOX, &tmBT, fb, n0 + j * 64, kb * BK, bz * bt.zb);
                }
                if (chunked & 2) {
                    tma_load_4d(sa + BT_STAGE, &tmA, fb, 0, 0, kb * (BK / 64), bz * bt.za);
                } else {
#pragma unroll
                    for (int j = 0; j < BK / 64; ++j)
                        tma_load_3d(sa + BT_STAGE + j * Cfg::A_ATOM, &tmA, fb, kb * BK + j * 64, 0,
                                    bz * bt.za);
                }
                ++issued;
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            int ds = s;
            uint32_t dph = ph;
            const uint32_t n_drain = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
            for (uint32_t i = 0; i < n_drain; ++i) {
                if (--ds < 0) {
                    ds = STAGES - 1;
                    dph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&full_bar[ds]), dph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // A operand = B^T tile (MN-major), B operand = A tile (K-major).
            constexpr uint32_t idesc = idesc_f16_f32(BNT, MP, true, false);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = base + s * Cfg::STAGE;
                const uint64_t btd = sdesc_sw128(sa, BK * 128, 1024);
                const uint64_t ad = sdesc_sw128(sa + BT_STAGE, 16, 1024);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_f16(tmem_base, btd + (k * 2048u >> 4),
                             ad + ((k / 4) * (Cfg::A_ATOM >> 4) + (k % 4) * 2), idesc,
                             (kb != kb0 || k != 0) ? 1u : 0u);
                umma_commit(smem_u32(&empty_bar[s]));
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_SKINNY);
            } else {
                umma_commit(smem_u32(&tfull_bar));
            }
            umma_commit(smem_u32(&drain_bar));
            if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else {
        // Accumulator -> this CTA's fp32 partial in shared memory, [MP][128]:
        // lane n of warp quadrant q holds the MP values of row n = 32q + lane.
        const int q = warp & 3;
        const bool got = mbar_wait(smem_u32(&tfull_bar), 0, &abort_flag, epi_limit);
        if (__all_sync(0xffffffffu, got)) {
            tc_fence_after();
            const int nl = q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
            for (int c = 0; c < MP; c += 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(taddr + c, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    red[(c + j) * BNT + nl] = (kb1 > kb0) ? __uint_as_float(r[j]) : 0.0f;
            }
        } else if (lane == 0) {
            abort_flag = 1;
            atomicOr(err, ERR_SKINNY);
        }
        tc_fence_before();
    }

    // All partials of the cluster are in shared memory after this barrier.
    cluster_sync();

    {
        // rows n this CTA reduces, four at a time: every CTA's partial of the
        // four is loaded (16 bytes each, all loads in flight together) before
        // they are added, in rank order
        const int span = BNT / split;
        const int quads = span / 4;
        const uint32_t red_local = smem_u32(red);
        for (int idx = threadIdx.x; idx < quads * M; idx += kThreads) {
            const int m = idx / quads;
            const int nl = rank * span + 4 * (idx - m * quads);
            if (n0 + nl >= N) continue;
            const uint32_t off = static_cast<uint32_t>((m * BNT + nl) * 4);
            float4 part[kMaxSplit];
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r)
                if (r < split) part[r] = ld_dsmem_f32x4(mapa_shared(red_local + off, static_cast<uint32_t>(r)));
            float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r) {
                if (r < split) {
                    sum[0] += part[r].x;
                    sum[1] += part[r].y;
                    sum[2] += part[r].z;
                    sum[3] += part[r].w;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + nl + j;
                if (n >= N) break;
                float y = sum[j];
                if (epi.on) y = epilogue_elem<OUT_F32>(y, m, n, epi);
                if constexpr (OUT_F32)
                    static_cast<float*>(Cb)[static_cast<long long>(m) * ldc + n] = y;
                else
                    static_cast<__half*>(Cb)[static_cast<long long>(m) * ldc + n] = __float2half_rn(y);
            }
        }
    }

    // No CTA may leave while a peer can still read its shared memory.
    pdl_trigger();  // this CTA has issued all its global writes
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

std::mutex g_mu;
bool g_attr_set[64][8];
// Clusters of 2, 4 and 8 CTAs that can be resident at once, per device and
// kernel instance (large clusters need whole free groups of SMs).
int g_max_clusters[64][8][3];

// Largest split s (1, 2, 4 or 8) such that n_tiles * s CTAs run as one wave
// of co-resident clusters and every CTA keeps at least two k-blocks.
int choose_split(long long n_tiles, int nkb, int num_sms, const int (&max_clusters)[3])
{
    int s = 1;
    for (int i = 0; i < 3; ++i) {
        const int t = 2 << i;
        if (t > kMaxSplit || n_tiles * t > num_sms || n_tiles > max_clusters[i] ||
            nkb < 2 * t)
            break;
        s = t;
    }
    return s;
}

template <int MP, bool OUT_F32>
cudaError_t launch_cfg(const GemmArgs& a)
{
    using Cfg = SkinnyCfg<MP>;
    auto kernel = gemm_skinny_kernel<MP, OUT_F32>;
    int split = 1;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        const int slot = (MP / 16 - 1) * 2 + (OUT_F32 ? 1 : 0);
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_attr_set[dev][slot]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(Cfg::SMEM));
            if (e != cudaSuccess) return e;
            for (int i = 0; i < 3; ++i) {
                cudaLaunchConfig_t q = {};
                q.gridDim = dim3(2 << i, 1);
                q.blockDim = dim3(kThreads);
                q.dynamicSmemBytes = Cfg::SMEM;
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
                g_max_clusters[dev][slot][i] = n;
            }
            g_attr_set[dev][slot] = true;
        }
        split = choose_split(static_cast<long long>((a.N + BNT - 1) / BNT) * a.batch,
                             (a.K + BK - 1) / BK, a.num_sms, g_max_clusters[dev][slot]);
    }
    CUtensorMap ta, tbt;
    // A's two k-blocks of 64 and B^T's two column blocks of 64 in one copy
    // each when K (for A) or N (for B^T) is a whole number of blocks
    const int chunked = (a.N % 64 == 0 ? 1 : 0) |
                        (a.K % 64 == 0 ? 2 : 0);
    if ((chunked & 2)
            ? !encode_tmap_chunks(&ta, a.A, 2, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                                  static_cast<uint64_t>(a.lda), a.batch, a.sA, 64, MP, BK / 64)
            : !encode_tmap(&ta, a.A, 2, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                           static_cast<uint64_t>(a.lda), a.batch, a.sA, 64, MP))
        return cudaErrorInvalidValue;
    if ((chunked & 1)
            ? !encode_tmap_chunks(&tbt, a.B, 2, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                                  static_cast<uint64_t>(a.ldb), a.batch, a.sB, 64, BK, BNT / 64)
            : !encode_tmap(&tbt, a.B, 2, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                           static_cast<uint64_t>(a.ldb), a.batch, a.sB, 64, BK))
        return cudaErrorInvalidValue;
    const int n_tiles = (a.N + BNT - 1) / BNT;
    if (n_tiles > 65535 || a.batch > 65535) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(split, n_tiles, a.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = a.stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = split;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    set_pdl_attr(at[1]);
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tbt, a.C, a.ldc, a.M, a.N, a.K, split, chunked,
                              a.hook, a.err, a.epi, a.batch_args());
}

}  // namespace

cudaError_t launch_skinny(const GemmArgs& a)
{
    if (a.M > kSkinnyMaxM) return cudaErrorInvalidValue;
    const int mp = (a.M + 15) / 16 * 16;
    if (a.out_f32) {
        switch (mp) {
            case 16: return launch_cfg<16, true>(a);
            case 32: return launch_cfg<32, true>(a);
            case 48: return launch_cfg<48, true>(a);
            default: return launch_cfg<64, true>(a);
        }
    }
    switch (mp) {
        case 16: return launch_cfg<16, false>(a);
        case 32: return launch_cfg<32, false>(a);
        case 48: return launch_cfg<48, false>(a);
        default: return launch_cfg<64, false>(a);
    }
}

}  // namespace tg

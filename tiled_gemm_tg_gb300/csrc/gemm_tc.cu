// gemm_tc.cu -- the one-CTA GEMM kernel for sm_103a: C = A x B (fp16 or
// E4M3 inputs) with fp32 accumulation in tensor memory, for mid-size,
// small-K and batched problems.
//
// What the pages describe ("企业官网建设流程全解析" (cf-1.com), §2.3 and §3.3):
// a 2-D grid of 128x128 output tiles, A and B tiles staged in shared memory,
// an fp32 accumulator cleared once per tile, the K loop software-pipelined
// over num_stages buffers (copy A, copy B, gemm), a swizzled shared-memory
// layout against bank conflicts (§4.1), and warp specialisation with a
// TMA producer feeding compute warps through mbarriers (§2.3).
//
// How it is built here for GB300:
//   * persistent grid of one CTA per SM walking a grouped tile order, so a
//     wave of tiles shares A rows and B columns in L2 (the "block_wise"
//     mapping of "TileLang：GPU异构计算的声明式分块编程范式" (kwkr.cn), §3.3);
//   * tiles of 128 x BN (BN = 256, 128 or 64), k-blocks of one 128-byte
//     swizzle atom per row (64 fp16 or 128 E4M3) for BN = 256 and of two
//     for BN = 128 or 64; a strided batch walks every tile of every matrix
//     through 3-D (or 4-D) tensor maps;
//   * warp 0: TMA producer.  A is loaded K-major ([128 rows][128 B]), B is
//     loaded MN-major in 128-byte-wide blocks of [k rows][128 B of n], all
//     with the 128-byte swizzle, into a ring of STAGES full/empty mbarrier
//     pairs; when N is a whole number of blocks one 4-D copy brings all
//     BN / 64 blocks of a stage (a copy costs about the same whatever its
//     size, so fewer, larger copies fill a stage sooner);
//   * warp 1: allocates tensor memory and issues tcgen05.mma (M=128, N=BN,
//     32 bytes of k each, four per k-block) from one thread, accumulating in
//     a double-buffered TMEM accumulator (2 x BN fp32 columns);
//   * warps 2..9: epilogue, two per TMEM lane quadrant (half of the columns
//     each).  Each thread owns one output row: tcgen05.ld of 32 columns at a
//     time, the fused epilogue if any, fp32 -> fp16 round-to-nearest-even
//     (or fp32 as is).  When C is TMA-addressable and its rows end on
//     16-byte boundaries the warp's 32 x 32 chunks go through a 4 KB
//     shared-memory staging buffer per warp (two fp16 chunks double-
//     buffered) and leave as one TMA store each (the TMA engine clips them
//     at the M/N edges); otherwise each thread writes its row with 16-byte
//     vector stores, predicated at the edges.  After its last TMEM read each
//     epilogue warp arrives on a named barrier on which warp 1 waits to free
//     TMEM, so the release overlaps the last stores.  The epilogue of tile i overlaps the main loop of tile i+1.
// A problem with few output tiles (at most half the SMs) is also split over
// K: a cluster of S CTAs (2, 4 or 8) shares each tile, CTA r taking k-blocks
// [r*nkb/S, (r+1)*nkb/S).  The epilogue warps then copy the accumulator into
// the CTA's own shared memory (fp32, rows padded by four floats so the
// copies from TMEM lanes do not collide on banks), the cluster
// synchronises, and all 320 threads of CTA r add up rows [r*128/S,
// (r+1)*128/S) of the S partials through distributed shared memory, in rank
// order, apply the fused epilogue and store them.
// Out-of-range rows, columns and k are zero-filled by TMA, so any M, N, K
// works as long as the operands are TMA-addressable (16-byte aligned bases,
// row strides a multiple of 16 bytes); the host routes everything else to
// the boundary kernel.
//
// Every mbarrier wait is bounded.  A role that gives up records a bit in the
// device error word and raises a shared abort flag; the other roles then
// give up too, the producer waits (bounded) for its own TMA copies in
// flight, the MMA thread waits for its own MMAs, and tensor memory is freed
// before the CTA exits.
#include <cstdint>
#include <cstring>
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

constexpr int BM = 128;
// 128-byte swizzle atoms of A per k-block: two for tiles of 64 or 128
// columns (stages of 48 or 64 KB, four or three deep), one for 256 columns
// (48 KB, four deep).  Measured in CUDA-graph replay against one atom
// everywhere: 1024 x 2048 x 512 5.51 against 6.35 us, 1024^3 6.42 against
// 8.45; with 256 columns two atoms (two stages of 96 KB) were slower
// (2048 x 2048 x 1024 11.6 against 10.3 us).
constexpr int katoms(int bn) { return bn == 256 ? 1 : 2; }
// A k-block is KATOMS x 128 bytes of every row: KATOMS atoms of 64 fp16 or
// 128 E4M3 elements (ES = element size in bytes), four MMAs of 32 bytes per
// atom.
template <int ES, int KATOMS>
struct KBlock {
    static constexpr int AE = 128 / ES;             // k elements per A atom
    static constexpr int BK = KATOMS * AE;          // k elements per k-block
    static constexpr int NB = 128 / ES;             // n elements per B box (128 bytes)
    static constexpr uint32_t B_BOX = BK * 128;     // one [BK k][NB n] box
    static constexpr uint32_t B_KSTEP = 32 / ES * 128 / 16;  // 16-byte units per MMA k step
};
constexpr uint32_t A_ATOM = BM * 128;
// Two epilogue warps per TMEM lane quadrant, each draining half of the
// accumulator's columns: a long fused epilogue (GELU) then keeps up with the
// MMAs instead of holding the accumulator buffer.
constexpr int kEpilogueWarps = 8;
constexpr int kThreads = 64 + 32 * kEpilogueWarps;
// Output staging for TMA stores: 4 KB per epilogue warp, one 32 x 32 fp32
// chunk or two fp16 chunks (double-buffered).
constexpr uint32_t kStageC = 4096;
constexpr uint32_t kStageCBytes = kEpilogueWarps * kStageC;
// Named barrier on which the epilogue warps tell warp 1 that their last
// TMEM read is done: the eight epilogue warps arrive, warp 1 waits.
constexpr int kTmemFreeBar = 1;
constexpr int kTmemFreeThreads = 32 * (kEpilogueWarps + 1);

// fp32 partial tile of a split over K: BM rows of BN + 4 floats.
template <int BN>
struct RedCfg {
    static constexpr int LD = BN + 4;
    static constexpr uint32_t BYTES = BM * LD * 4;
};
constexpr int kMaxSplitK = 8;

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t cluster_addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

template <int BN>
struct MainCfg {
    static constexpr int KATOMS = katoms(BN);
    static constexpr uint32_t A_STAGE = KATOMS * A_ATOM;
    static constexpr uint32_t B_STAGE = BN * 128 * KATOMS;
    static constexpr uint32_t STAGE = A_STAGE + B_STAGE;
    // the most stages that fit (the default); a ring of 2..STAGES can be
    // requested (tg_gemm_force_stages), shared memory is sized to it
    static constexpr int STAGES = (BN == 256 ? 4 : (BN == 128 ? 6 : 8)) / KATOMS;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr uint32_t SMEM = STAGES * STAGE + 1024;  // + alignment slack
    static constexpr uint32_t smem(int stages, bool c_tma)
    {
        return stages * STAGE + (c_tma ? kStageCBytes : 0u) + 1024;
    }
    static_assert(SMEM + kStageCBytes <= 227 * 1024, "shared-memory budget exceeded");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
};

template <int BN, bool OUT_F32, int ES>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_main_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, void* C, long long ldc, int M,
                    int N, int K, int tiles_m, int tiles_n, int group_m, int stages, int c_vec,
                    int c_tma, int split, int b_chunks, int a_chunks, int hook, unsigned int* err,
                    Epilogue epi,
                    BatchArgs bt)
{
    using Cfg = MainCfg<BN>;
    constexpr int STAGES = Cfg::STAGES;  // the most stages; `stages` are in use

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 32 * kEpilogueWarps);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    constexpr int KATOMS = Cfg::KATOMS;
    using KB = KBlock<ES, KATOMS>;
    constexpr int BK = KB::BK;
    constexpr int NB = KB::NB;
    constexpr uint32_t B_BOX = KB::B_BOX;
    constexpr uint32_t A_STAGE = Cfg::A_STAGE;
    static_assert(BN % NB == 0, "B tile must be whole 128-byte boxes");
    // a split over K: this CTA is rank r of a cluster of `split` sharing one
    // tile, and takes k-blocks kb_lo .. kb_lo + num_kb - 1 of it
    // (the divisions are kept off the unsplit kernel's path to its first
    // load: a 64-bit division alone costs ~100 instructions)
    const int total = tiles_m * tiles_n * bt.count;
    int rank = 0, kb_lo = 0, num_kb = (K + BK - 1) / BK;
    // the tiles this CTA walks: t_first, t_first + t_step, ... (one tile when split)
    int t_first = static_cast<int>(blockIdx.x), t_step = static_cast<int>(gridDim.x);
    if (split > 1) {
        const int nkb_all = num_kb;  // < 2^25, so rank * nkb_all fits in an int
        rank = static_cast<int>(cluster_ctarank());
        kb_lo = rank * nkb_all / split;
        num_kb = (rank + 1) * nkb_all / split - kb_lo;
        t_first = static_cast<int>(blockIdx.x) / split;
        t_step = total;
    }
    // the producer's first tile, found before the wait for the previous
    // kernel (the integer divisions of the tile order are on the critical
    // path of a one-tile CTA otherwise)
    int b0 = 0, tm0 = 0, tn0 = 0;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        // the first tile's first stages into L2 while the previous kernel finishes
        if (t_first < total) {
            batch_tile_coords(t_first, tiles_m, tiles_n, group_m, b0, tm0, tn0);
            const int b = b0, tm = tm0, tn = tn0;
            const int pf = total > t_step ? stages : min(stages, kPrefetchStagesSingle);
            for (int kb = 0; kb < num_kb && kb < pf; ++kb) {
                if (a_chunks) {
                    tma_prefetch_l2_4d(&tmA, 0, tm * BM, (kb_lo + kb) * KATOMS, b * bt.za);
                } else {
                    for (int j = 0; j < KATOMS; ++j)
                        tma_prefetch_l2_3d(&tmA, (kb_lo + kb) * BK + j * KB::AE, tm * BM,
                                           b * bt.za);
                }
                if (b_chunks) {
                    tma_prefetch_l2_4d(&tmB, 0, (kb_lo + kb) * BK, tn * (BN / NB), b * bt.zb);
                } else {
                    for (int j = 0; j < BN / NB; ++j)
                        tma_prefetch_l2_3d(&tmB, tn * BN + j * NB, (kb_lo + kb) * BK, b * bt.zb);
                }
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

    // The epilogue waits for a whole tile's main loop; allow ~64 us per k-block
    // on top of the base limit so long-K problems never time out spuriously.
    const uint32_t epi_limit = kSlowPolls + 64u * static_cast<uint32_t>(min(num_kb, 1 << 20));

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            for (int t = t_first; t < total; t += t_step) {
                int b = b0, tm = tm0, tn = tn0;
                if (t != t_first)
                    batch_tile_coords(t, tiles_m, tiles_n, group_m, b, tm, tn);
                const int za = b * bt.za, zb = b * bt.zb;
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, &abort_flag)) {
                        abort_flag = 1;
                        atomicOr(err, ERR_MAIN_PRODUCER);
                        ok = false;
                        break;
                    }
                    if (hook == 1 && t == t_first && kb == 0) {
                        // test hook: leave this stage unfilled, so the MMA
                        // thread's bounded wait on it runs out
                        if (++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    const uint32_t fb = smem_u32(&full_bar[s]);
                    const uint32_t sa = base + s * Cfg::STAGE;
                    mbar_arrive_expect_tx(fb, Cfg::STAGE);
                    if (a_chunks) {
                        tma_load_4d(sa, &tmA, fb, 0, tm * BM, (kb_lo + kb) * KATOMS, za);
                    } else {
#pragma unroll
                        for (int j = 0; j < KATOMS; ++j)
                            tma_load_3d(sa + j * A_ATOM, &tmA, fb,
                                        (kb_lo + kb) * BK + j * KB::AE, tm * BM, za);
                    }
                    if (b_chunks) {
                        // all BN / NB column blocks of B in one copy
                        tma_load_4d(sa + A_STAGE, &tmB, fb, 0, (kb_lo + kb) * BK, tn * (BN / NB),
                                    zb);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / NB; ++j)
                            tma_load_3d(sa + A_STAGE + j * B_BOX, &tmB, fb, tn * BN + j * NB,
                                        (kb_lo + kb) * BK, zb);
                    }
                    ++issued;
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // Wait for this thread's own copies still in flight: the most
            // recent arming of each of the last min(issued, stages) stages.
            int ds = s;
            uint32_t dph = ph;
            const uint32_t n_drain = issued < (uint32_t)stages ? issued : (uint32_t)stages;
            for (uint32_t i = 0; i < n_drain; ++i) {
                if (--ds < 0) {
                    ds = stages - 1;
                    dph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&full_bar[ds]), dph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN, false, true);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (int t = t_first; t < total && ok; t += t_step) {
                if (!mbar_wait(smem_u32(&tempty_bar[acc]), aph ^ 1u, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * Cfg::STAGE;
                    // A: K-major, 8-row groups 1024 B apart, +32 B per MMA.  B:
                    // MN-major, 128-byte-wide boxes B_BOX apart, 8-row k groups
                    // 1024 B apart, one MMA's k rows (16 fp16 / 32 E4M3) per step.
                    const uint64_t ad = sdesc_sw128(sa, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sa + A_STAGE, B_BOX, 1024);
#pragma unroll
                    for (int k = 0; k < 4 * KATOMS; ++k)
                        umma<ES>(d, ad + ((k / 4) * (A_ATOM >> 4) + (k % 4) * 2ull),
                                 bd + KB::B_KSTEP * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(smem_u32(&empty_bar[s]));
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull_bar[acc]));
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_MAIN_MMA);
            }
            // Every MMA this thread issued must finish before TMEM is freed.
            umma_commit(smem_u32(&drain_bar));
            if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        constexpr int span = BN / (kEpilogueWarps / 4);  // accumulator columns per warp
        const int c_lo = ((warp - 2) >> 2) * span;
        const uint32_t stage_c = base + static_cast<uint32_t>(stages) * Cfg::STAGE +
                                 static_cast<uint32_t>(warp - 2) * kStageC;
        uint32_t chunk = 0;  // staged chunks so far (fp16 alternates two 2 KB halves)
        int acc = 0;
        uint32_t aph = 0;
        if (split > 1) {
            // the accumulator (this CTA's k-range of its one tile) -> the fp32
            // partial in shared memory, row q*32 + lane at red[row * LD]; the
            // stages are free once every MMA is complete
            const bool got = mbar_wait(smem_u32(&tfull_bar[0]), 0, &abort_flag, epi_limit);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                float* const red = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
                const int ml = q * 32 + lane;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
                for (int c = c_lo; c < c_lo + span; c += 32) {
                    uint32_t r[32];
                    if (num_kb > 0) {
                        tmem_ld_32x32b_x32(taddr + c, r);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    float4* row = reinterpret_cast<float4*>(red + ml * RedCfg<BN>::LD + c);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        row[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                             __uint_as_float(r[4 * j + 2]),
                                             __uint_as_float(r[4 * j + 3]));
                }
            } else if (lane == 0) {
                abort_flag = 1;
                atomicOr(err, ERR_MAIN_EPILOGUE);
            }
        }
        for (int t = t_first; t < total && split == 1; t += t_step) {
            int b, tm, tn;
            batch_tile_coords(t, tiles_m, tiles_n, group_m, b, tm, tn);
            void* Cb = batch_ptr(C, b, bt.sC, OUT_F32 ? 4 : 2);
            const bool got = mbar_wait(smem_u32(&tfull_bar[acc]), aph, &abort_flag, epi_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    abort_flag = 1;
                    atomicOr(err, ERR_MAIN_EPILOGUE);
                }
                break;
            }
            tc_fence_after();
            const int m0 = tm * BM + q * 32;  // this warp's first row
            const int m = m0 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = c_lo; c < c_lo + span; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c, r);
                tmem_ld_wait();
                const int n = tn * BN + c;
                if (c_tma) {
                    if (m0 < M && n < N) {  // warp-uniform
                        if (epi.on && m < M) epilogue_chunk<OUT_F32>(r, m, n, N, epi);
                        // the staging buffer half (fp16) or whole (fp32) this
                        // chunk takes is free once the store that used it
                        // last has read it
                        if (lane == 0) {
                            if constexpr (OUT_F32) bulk_wait_read<0>();
                            else bulk_wait_read<1>();
                        }
                        __syncwarp();
                        const uint32_t slot = OUT_F32 ? stage_c : stage_c + (chunk & 1u) * (kStageC / 2);
                        stage_store_chunk<OUT_F32>(&tmC, slot, r, n, m0, b, lane);
                        ++chunk;
                    }
                } else if (m < M && n < N) {
                    if (epi.on) epilogue_chunk<OUT_F32>(r, m, n, N, epi);
                    store_chunk<OUT_F32>(Cb, ldc, m, n, N, r, c_vec != 0);
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty_bar[acc]));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        // every TMEM read of this warp is done: warp 1 may free TMEM now,
        // while the last stores drain
        tc_fence_before();
        named_bar_arrive(kTmemFreeBar, kTmemFreeThreads);
        // the TMA stores have read their staging buffers before the CTA
        // ends (their writes to C complete with the grid)
        if (c_tma && lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }

    if (split > 1) {
        if (warp == 1) {
            named_bar_sync(kTmemFreeBar, kTmemFreeThreads);
            tc_fence_after();
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
        }
        // every partial of the cluster is in shared memory after this barrier
        cluster_sync();
        if (t_first < total) {
            int b, tm, tn;
            batch_tile_coords(t_first, tiles_m, tiles_n, group_m, b, tm, tn);
            void* Cb = batch_ptr(C, b, bt.sC, OUT_F32 ? 4 : 2);
            // rows rank*rows .. of the tile, four columns per item, every
            // thread of the CTA; the partials are added in rank order
            const int rows = BM / split;
            constexpr int quads = BN / 4;
            for (int idx = threadIdx.x; idx < rows * quads; idx += kThreads) {
                const int ml = rank * rows + idx / quads;
                const int nl = 4 * (idx % quads);
                const int m = tm * BM + ml, n = tn * BN + nl;
                if (m >= M || n >= N) continue;
                const uint32_t off = static_cast<uint32_t>((ml * RedCfg<BN>::LD + nl) * 4);
                float4 part[kMaxSplitK];
#pragma unroll
                for (int r = 0; r < kMaxSplitK; ++r)
                    if (r < split) part[r] = ld_cluster_f32x4(mapa_shared(base + off, static_cast<uint32_t>(r)));
                float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int r = 0; r < kMaxSplitK; ++r) {
                    if (r < split) {
                        v[0] += part[r].x;
                        v[1] += part[r].y;
                        v[2] += part[r].z;
                        v[3] += part[r].w;
                    }
                }
                const bool full = n + 4 <= N;
                if (epi.on) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n + j < N) v[j] = epilogue_elem<OUT_F32>(v[j], m, n + j, epi);
                }
                if constexpr (OUT_F32) {
                    float* row = static_cast<float*>(Cb) + static_cast<long long>(m) * ldc + n;
                    if (c_vec && full) {
                        *reinterpret_cast<float4*>(row) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (n + j < N) row[j] = v[j];
                    }
                } else {
                    __half* row = static_cast<__half*>(Cb) + static_cast<long long>(m) * ldc + n;
                    if (c_vec && full) {
                        const __half2 lo = __floats2half2_rn(v[0], v[1]);
                        const __half2 hi = __floats2half2_rn(v[2], v[3]);
                        *reinterpret_cast<uint2*>(row) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                       *reinterpret_cast<const uint32_t*>(&hi));
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (n + j < N) row[j] = __float2half_rn(v[j]);
                    }
                }
            }
        }
        pdl_trigger();  // this CTA has issued all its global writes
        // no CTA may leave while a peer can still read its partial
        cluster_sync();
        return;
    }
    pdl_trigger();  // this CTA has issued all its global writes
    if (warp == 1) {
        // after the MMA thread's own MMAs (drained above) and every epilogue
        // warp's last TMEM read
        named_bar_sync(kTmemFreeBar, kTmemFreeThreads);
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

std::mutex g_attr_mu;
bool g_attr_set[64][12];
// Clusters of 2, 4 and 8 CTAs that fit at once, per device and kernel
// instance (with the default ring's shared memory).
int g_max_clusters[64][12][3];

// Clusters of S CTAs per tile for `tiles` tiles of nkb k-blocks: none when
// the tiles fill more than half of the SMs; else the largest S of 2, 4, 8
// with tiles * S <= num_sms, S <= nkb and (given max_clusters) all the
// clusters resident at once.
int main_split_k(long long tiles, long long nkb, int num_sms, const int* max_clusters)
{
    if (tiles * 2 > num_sms) return 1;
    int s = 1;
    for (int i = 0; i < 3; ++i) {
        const int t = 2 << i;
        if (tiles * t > num_sms || nkb < t || (max_clusters != nullptr && tiles > max_clusters[i]))
            break;
        s = t;
    }
    return s;
}

// The kernel instance's launch attributes, set once per device, and its
// cluster residency: max_clusters[i] clusters of 2 << i CTAs fit at once.
template <int BN, bool OUT_F32, int ES>
cudaError_t init_instance(const int** max_clusters)
{
    using Cfg = MainCfg<BN>;
    auto kernel = gemm_tc_main_kernel<BN, OUT_F32, ES>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int slot =
        ((BN == 256 ? 0 : BN == 128 ? 1 : 2) * 2 + (OUT_F32 ? 1 : 0)) * 2 + (ES == 1 ? 1 : 0);
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (!g_attr_set[dev][slot]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg::SMEM + kStageCBytes));
        if (e != cudaSuccess) return e;
        for (int i = 0; i < 3; ++i) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2 << i);
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
    *max_clusters = g_max_clusters[dev][slot];
    return cudaSuccess;
}

template <bool OUT_F32, int ES>
cudaError_t instance_clusters(int bn, const int** mc)
{
    if (bn == 256) return init_instance<256, OUT_F32, ES>(mc);
    if constexpr (ES == 1) {
        return init_instance<128, OUT_F32, ES>(mc);  // E4M3 tiles are 128 or 256 wide
    } else {
        if (bn == 128) return init_instance<128, OUT_F32, ES>(mc);
        return init_instance<64, OUT_F32, ES>(mc);
    }
}

cudaError_t clusters_of(const GemmArgs& a, int bn, const int** mc)
{
    if (a.in_es == 1)
        return a.out_f32 ? instance_clusters<true, 1>(bn, mc) : instance_clusters<false, 1>(bn, mc);
    return a.out_f32 ? instance_clusters<true, 2>(bn, mc) : instance_clusters<false, 2>(bn, mc);
}

// Estimated microseconds of a call with tile width bn split s ways over K,
// from sweeps of every tile width and split on GB300 (CUDA-graph replay,
// operands past L2): each CTA takes in A and B at ~100 KB/us on its own and
// ~110 KB/us in a split with k-blocks of two atoms (64- and 128-column
// tiles), ~86 and ~95 KB/us with one (256 columns), times the waves when the
// CTAs outnumber the SMs; a split adds ~1.5, 2.5 or 4.0 us for 64, 128 or
// 256 columns (the partial tile through distributed shared memory and the
// two cluster barriers).
double main_cost_us(long long M, long long N, long long K, long long batch, int es, int num_sms,
                    int bn, int s)
{
    const int bk = katoms(bn) * 128 / es;
    const long long tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn) * batch;
    const long long waves = (tiles * s + num_sms - 1) / num_sms;
    const long long nkb = (K + bk - 1) / bk;
    // the k-range of one CTA (a k-block past K is zero fill, not bytes)
    long long kper = (nkb + s - 1) / s * bk;
    if (kper > K) kper = K;
    const long long rows = M < BM ? M : BM;
    const long long n64 = (N + 63) / 64 * 64;
    const long long cols = n64 < bn ? n64 : bn;
    const double kbytes = static_cast<double>((rows + cols) * kper * es) / 1024.0;
    const bool two = katoms(bn) == 2;
    if (s == 1) return static_cast<double>(waves) * kbytes / (two ? 100.0 : 86.0);
    const double extra = bn == 64 ? 1.5 : bn == 128 ? 2.5 : 4.0;
    return static_cast<double>(waves) * kbytes / (two ? 110.0 : 95.0) + extra;
}

// The tile width and split for a call (max_clusters(bn) gives the residency
// of each instance, or null for the rule alone).  A forced split is used as
// given (halved while it exceeds the k-blocks); otherwise the default tile
// width, unsplit, competes with every other width unsplit and every width
// at its largest split, by estimated time.
template <typename MC>
void plan(long long M, long long N, long long K, long long batch, int es, int num_sms,
          int forced_bn, int forced_split, MC max_clusters, int* bn_out, int* split_out)
{
    int bn = forced_bn != 0 ? forced_bn
                            : main_tile_n(static_cast<int>(M), static_cast<int>(N),
                                          static_cast<int>(batch), num_sms);
    if (es == 1 && bn == 64) bn = 128;  // E4M3 B boxes are 128 elements wide
    // k-blocks of a tile width
    auto nkb_of = [&](int w) { return (K + katoms(w) * 128 / es - 1) / (katoms(w) * 128 / es); };
    int split = 1;
    if (forced_split > 0) {
        split = forced_split;
        while (split > 1 && split > nkb_of(bn)) split >>= 1;
    } else {
        // another width or a split must be estimated 5 % faster than the
        // default width, unsplit, to replace it
        double best = 0.95 * main_cost_us(M, N, K, batch, es, num_sms, bn, 1);
        const int widths[3] = {64, 128, 256};
        for (int w : widths) {
            if ((forced_bn != 0 && w != forced_bn) || (es == 1 && w == 64)) continue;
            const long long tiles = ((M + BM - 1) / BM) * ((N + w - 1) / w) * batch;
            const int sw = main_split_k(tiles, nkb_of(w), num_sms, max_clusters(w));
            const int tries[2] = {1, sw};
            for (int sp : tries) {
                if (sp == 1 && w == bn) continue;
                const double c = main_cost_us(M, N, K, batch, es, num_sms, w, sp);
                if (c < best) {
                    best = c;
                    bn = w;
                    split = sp;
                }
            }
        }
    }
    *bn_out = bn;
    *split_out = split;
}

template <int BN, bool OUT_F32, int ES>
cudaError_t launch_cfg(const GemmArgs& a)
{
    using Cfg = MainCfg<BN>;
    using KB = KBlock<ES, Cfg::KATOMS>;
    constexpr int KATOMS = Cfg::KATOMS;
    auto kernel = gemm_tc_main_kernel<BN, OUT_F32, ES>;
    const int* mc = nullptr;
    {
        const cudaError_t e = init_instance<BN, OUT_F32, ES>(&mc);
        if (e != cudaSuccess) return e;
    }
    const int split = a.split_k > 1 ? a.split_k : 1;
    CUtensorMap ta, tb;
    // A's KATOMS atoms of a k-block in one copy when K is a whole number of
    // atoms
    const int a_chunks = KATOMS > 1 && a.K % KB::AE == 0 ? 1 : 0;
    if (a_chunks ? !encode_tmap_chunks(&ta, a.A, ES, static_cast<uint64_t>(a.K),
                                       static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda),
                                       a.batch, a.sA, KB::AE, BM, KATOMS)
                 : !encode_tmap(&ta, a.A, ES, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                                static_cast<uint64_t>(a.lda), a.batch, a.sA, KB::AE, BM))
        return cudaErrorInvalidValue;
    // B's BN / NB column blocks of a k-block in one copy when N is a whole
    // number of blocks (a block past N would read beyond the matrix)
    const int b_chunks = BN > KB::NB && a.N % KB::NB == 0 ? 1 : 0;
    if (b_chunks) {
        if (!encode_tmap_chunks(&tb, a.B, ES, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                                static_cast<uint64_t>(a.ldb), a.batch, a.sB, KB::NB, KB::BK,
                                BN / KB::NB))
            return cudaErrorInvalidValue;
    } else if (!encode_tmap(&tb, a.B, ES, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                            static_cast<uint64_t>(a.ldb), a.batch, a.sB, KB::NB, KB::BK)) {
        return cudaErrorInvalidValue;
    }
    const int tiles_m = (a.M + BM - 1) / BM;
    const int tiles_n = (a.N + BN - 1) / BN;
    const int total = tiles_m * tiles_n * a.batch;
    const int grid = total < a.num_sms ? total : a.num_sms;
    const int group_m = a.group_m > 0 ? a.group_m : 16;
    const size_t es = OUT_F32 ? 4 : 2;
    const int c_vec = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) &&
                      ((static_cast<size_t>(a.ldc) * es) % 16 == 0) &&
                      ((static_cast<size_t>(a.sC) * es) % 16 == 0);
    // C written by TMA stores (32 x 32 boxes) when the TMA engine can
    // address it and each row of C ends on a 16-byte boundary: at the right
    // edge of C a TMA store writes whole 16-byte units (measured: a box
    // clipped at N = 129 fp32 columns also wrote columns 129..131 of the row
    // stride), and the ABI leaves columns N..ldc-1 untouched
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    // (a split over K stores from its reduction, without TMA)
    const int c_tma = split == 1 && c_vec && (static_cast<size_t>(a.N) * es) % 16 == 0 &&
                      encode_tmap_store(&tc, a.C, static_cast<int>(es),
                                        static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M),
                                        static_cast<uint64_t>(a.ldc), a.batch, a.sC, 32, 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(split > 1 ? total * split : grid);
    cfg.blockDim = dim3(kThreads);
    const int stages = a.stages > 0 ? a.stages : Cfg::STAGES;
    if (stages < 2 || stages > Cfg::STAGES) return cudaErrorInvalidValue;
    uint32_t smem = Cfg::smem(stages, c_tma != 0);
    if (split > 1 && smem < RedCfg<BN>::BYTES + 1024) smem = RedCfg<BN>::BYTES + 1024;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute at[2];
    set_pdl_attr(at[0]);
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = split;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = split > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, a.C, a.ldc, a.M, a.N, a.K, tiles_m,
                              tiles_n, group_m, stages, c_vec, c_tma, split, b_chunks, a_chunks,
                              a.hook, a.err, a.epi, a.batch_args());
}

}  // namespace

cudaError_t main_plan(const GemmArgs& a, int forced_bn, int forced_split, int* bn, int* split)
{
    cudaError_t err = cudaSuccess;
    auto mc = [&](int w) -> const int* {
        const int* p = nullptr;
        const cudaError_t e = clusters_of(a, w, &p);
        if (e != cudaSuccess) err = e;
        return p;
    };
    plan(a.M, a.N, a.K, a.batch, a.in_es, a.num_sms, forced_bn, forced_split, mc, bn, split);
    return err;
}

void main_plan_host(long long M, long long N, long long K, long long batch, int es, int num_sms,
                    int* bn, int* split)
{
    plan(M, N, K, batch, es, num_sms, 0, 0, [](int) -> const int* { return nullptr; }, bn, split);
}

int main_max_stages(int bn)
{
    return bn == 256 ? MainCfg<256>::STAGES : bn == 128 ? MainCfg<128>::STAGES : MainCfg<64>::STAGES;
}

int main_tile_n(int M, int N, int batch, int num_sms)
{
    const long long tm = static_cast<long long>((M + BM - 1) / BM) * batch;
    int w = 64;
    if (tm * ((N + 255) / 256) >= num_sms) w = 256;
    else if (tm * ((N + 127) / 128) >= num_sms / 2) w = 128;
    // never wider than N needs: columns past N only multiply zeros (a batch
    // of 64-column products in 256-column tiles ran at 0.70x the speed)
    const int cap = N <= 64 ? 64 : N <= 128 ? 128 : 256;
    return w < cap ? w : cap;
}

cudaError_t launch_main(const GemmArgs& a, int bn)
{
    if (a.in_es == 1) {
        // E4M3: B boxes are 128 elements wide, so tiles are 128 or 256 wide
        if (a.out_f32) return bn == 256 ? launch_cfg<256, true, 1>(a) : launch_cfg<128, true, 1>(a);
        return bn == 256 ? launch_cfg<256, false, 1>(a) : launch_cfg<128, false, 1>(a);
    }
    if (a.out_f32) {
        if (bn == 256) return launch_cfg<256, true, 2>(a);
        if (bn == 128) return launch_cfg<128, true, 2>(a);
        return launch_cfg<64, true, 2>(a);
    }
    if (bn == 256) return launch_cfg<256, false, 2>(a);
    if (bn == 128) return launch_cfg<128, false, 2>(a);
    return launch_cfg<64, false, 2>(a);
}

}  // namespace tg

// gemm_tc2.cu -- CTA-pair GEMM kernel for sm_103a: C = A x B (fp16 or E4M3
// inputs) with 256 x 256 output tiles computed by two CTAs of a cluster that
// share one tcgen05.mma.cta_group::2 (M=256, N=256, 32 bytes of k).
//
// The method is the pages' pipelined tiled GEMM ("企业官网建设流程全解析"
// (cf-1.com), §2.3 warp specialisation + TMA + mbarrier, §3.3 the tiled
// K loop with num_stages buffers, §4.1 swizzled shared memory); this file is
// the GB300 form of it for large problems.
//
// Why a pair: each CTA holds half of A's rows (128 rows x 256 B) and half of
// B's columns (256 B of k x 128 columns) of a 256 x 256 k-block, so a 64 KB
// stage feeds 1024 MMA cycles and each B column block is loaded once per pair
// instead of once per 128 rows (a third less L2 -> SM traffic than 128 x 256
// tiles).  Three stages fill 192 KB of shared memory.  When the last wave of
// tiles is at most half full, its tiles are cut into two 256 x 128 halves
// (work_item), each pair loading one 64-column B box per CTA and issuing
// N = 128 MMAs.  Each pair walks K forwards on its even-numbered tiles and
// backwards on its odd-numbered ones: the pairs of one wave share A rows with
// the wave before, whose last-read k-blocks are the ones still in L2 (8192^3:
// 1020 -> 854 MB of DRAM reads per launch, ~1 % faster).
//
// Roles (320 threads per CTA, the same in both CTAs of the pair):
//   warp 0   TMA producer.  Each CTA loads its own halves into its own shared
//            memory (a k-block's two A atoms, and its two B column blocks,
//            in one 4-D copy each when K, and N, are whole numbers of
//            blocks); every copy signals the EVEN (leader) CTA's full
//            barrier, which the leader's producer arms with both CTAs' bytes.
//   warp 1   both CTAs allocate 512 TMEM columns together (two 256-column
//            accumulators); only the leader's lane 0 issues the MMAs.  Each
//            k-block's commit is multicast to both CTAs' empty barriers,
//            each tile's commit to both CTAs' tmem-full barriers.
//   warps 2-9  epilogue in both CTAs, two per TMEM lane quadrant: each CTA
//            reads its own 128 rows of the accumulator from its own TMEM
//            (each warp half of the columns) and stores them, boxes of 32
//            rows x 128 bytes staged in shared memory and written by TMA
//            stores when C allows (16-byte aligned, rows ending on 16-byte
//            boundaries), else 16-byte stores per row; all epilogue threads
//            of the pair arrive on the leader's tmem-empty barrier.
// Waits are bounded as in the one-CTA kernel; on expiry a role records a bit
// in the device error word and leaves its loop; the leader waits for the
// pair's copies in flight and its own MMAs; a cluster barrier keeps both CTAs
// resident until then, and TMEM is freed by both CTAs together.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

using namespace tg::dev;

constexpr int PM = 256;                          // pair tile rows (128 per CTA)
constexpr int PN = 256;                          // pair tile columns (B: 128 per CTA)
constexpr int HM = PM / 2;
constexpr int HN = PN / 2;
// k-block of 256 bytes per row (128 fp16 or 256 E4M3 elements): eight MMAs
// of 32 bytes per stage and per commit.  Measured on GB300, 64-element fp16
// k-blocks (four MMAs between stage switches/commits) keep the tensor pipe
// 87-94 % busy, 128-element ones 100 %.
constexpr int KA = 2;                            // 128-byte swizzle atoms along k in A
constexpr uint32_t A_ATOM = HM * 128;            // [128 rows][128 bytes of k] = 16 KB
constexpr uint32_t A_STAGE = HM * 256;           // 32 KB
constexpr uint32_t B_STAGE = HN * 256;           // 32 KB
constexpr uint32_t STAGE = A_STAGE + B_STAGE;    // 64 KB per CTA

// Element-size dependent geometry (ES = 2: fp16, 1: E4M3).
template <int ES>
struct PairK {
    static constexpr int BK = 256 / ES;                  // k elements per k-block
    static constexpr int AE = 128 / ES;                  // k elements per A atom
    static constexpr int NB = 128 / ES;                  // n elements per B box
    static constexpr uint32_t B_BOX = BK * 128;          // one [BK k][NB n] box
    static constexpr uint32_t B_KSTEP = 32 / ES * 128 / 16;  // 16-byte units per MMA
};
// three 64 KB stages fit (the default); two can be requested
// (tg_gemm_force_stages), shared memory is sized to the ring
constexpr int STAGES = 3;
constexpr uint32_t SMEM = STAGES * STAGE + 1024;
// Output staging for TMA stores: 4 KB per epilogue warp (one box of 32 rows
// x 128 bytes), after the stages.
constexpr uint32_t kStageC = 4096;
constexpr uint32_t TMEM_COLS = 2 * PN;           // two accumulators
#ifndef TG_PAIR_EPI_WARPS
#define TG_PAIR_EPI_WARPS 8
#endif
// Epilogue warps: 4 (one per TMEM lane quadrant, each draining all 256
// accumulator columns of its 32 rows) or 8 (two per quadrant, 128 columns
// each).  Measured on 8192^3 bursts: the same 1800 TFLOP/s for the plain
// store, and 1714 instead of 1617 TFLOP/s with a GELU epilogue.
constexpr int EPI_WARPS = TG_PAIR_EPI_WARPS;
static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "4 or 8 epilogue warps");
constexpr uint32_t kEpilogueThreads = 32 * EPI_WARPS;
constexpr int kThreads = 64 + static_cast<int>(kEpilogueThreads);
constexpr int EPI_SPAN = PN / (EPI_WARPS / 4);  // accumulator columns per epilogue warp
constexpr uint32_t kStageCBytes = (kThreads / 32 - 2) * kStageC;
static_assert(SMEM + kStageCBytes <= 227 * 1024, "shared-memory budget exceeded");
static_assert(TMEM_COLS == 512, "two 256-column accumulators fill TMEM");
#ifndef TG_PAIR_L2_HINTS
#define TG_PAIR_L2_HINTS 1
#endif
constexpr int L2_HINTS = TG_PAIR_L2_HINTS;  // bit 0: A evict_last, bit 1: B evict_first

#ifndef TG_PAIR_EPI_COLS
#define TG_PAIR_EPI_COLS 32
#endif
constexpr int EPI_COLS = TG_PAIR_EPI_COLS;  // accumulator columns per tcgen05.ld

// Work item t of the pair kernel: tile t in the grouped order over the
// whole batch (half = -1), or, among the last `split_tail` tiles, one half
// of a tile: items past the whole tiles go two to a tile, half 0 for its
// columns 0..127 and half 1 for 128..255.  fp16 only (an E4M3 half would
// need a 64-byte-wide B box).
template <int ES>
__device__ __forceinline__ void work_item(int t, int tiles_m, int tiles_n, int group_m, int whole,
                                          int split_tail, int& b, int& tm, int& tn, int& half)
{
    half = -1;
    int tile = t;
    if (ES == 2 && split_tail > 0) {
        const int first = whole - split_tail;  // the first tile cut in two
        if (t >= first) {
            const int h = t - first;
            tile = first + (h >> 1);
            half = h & 1;
        }
    }
    batch_tile_coords(tile, tiles_m, tiles_n, group_m, b, tm, tn);
}

template <bool OUT_F32, int ES>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB4,
                    const __grid_constant__ CUtensorMap tmC, void* C, long long ldc, int M,
                    int N, int K, int tiles_m, int tiles_n, int group_m, int split_tail,
                    int stages, int c_vec, int c_tma, int chunked, int hook, unsigned int* err,
                    Epilogue epi, BatchArgs bt)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];   // used in the leader only
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];      // used in the leader only
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int npairs = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 2 * kEpilogueThreads);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (chunked & 1) tma_prefetch_desc(&tmB4);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    pdl_wait();  // the previous kernel on the stream is complete from here on

    using KG = PairK<ES>;
    constexpr int BK = KG::BK;
    const int num_kb = (K + BK - 1) / BK;
    // Work items: the tiles in the grouped order, except that the last
    // split_tail tiles (a short last wave) are each cut into two 256 x 128
    // halves, two items each, so that twice as many pairs share that wave.
    const int whole = tiles_m * tiles_n * bt.count;
    const int total = whole + (ES == 2 ? split_tail : 0);
    const uint32_t epi_limit = kSlowPolls + 64u * static_cast<uint32_t>(min(num_kb, 1 << 20));

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);  // leader's ring
            // L2 priorities: a group's A row blocks are reused by every wave of
            // the group, each B column block only by the tiles of one wave.
            const uint64_t pol_a = L2_HINTS & 1 ? policy_evict_last() : policy_evict_normal();
            const uint64_t pol_b = L2_HINTS & 2 ? policy_evict_first() : policy_evict_normal();
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = true;
            int wave = 0;
            for (int t = pair; t < total && ok; t += npairs, ++wave) {
                int b, tm, tn, half;
                work_item<ES>(t, tiles_m, tiles_n, group_m, whole, split_tail, b, tm, tn, half);
                // every other wave walks K backwards, starting on the k-blocks
                // of the A rows the wave before it read last (still in L2)
                const bool back = (wave & 1) != 0;
                const int za = b * bt.za, zb = b * bt.zb;
                const int row = tm * PM + static_cast<int>(rank) * HM;
                // a half item: each CTA holds 64 of its 128 columns (one box)
                const int col = half < 0 ? tn * PN + static_cast<int>(rank) * HN
                                         : tn * PN + half * HN + static_cast<int>(rank) * (HN / 2);
                const int nbox = half < 0 ? HN / KG::NB : 1;
                const uint32_t stage_bytes = A_STAGE + static_cast<uint32_t>(nbox) * KG::B_BOX;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, &abort_flag)) {
                        abort_flag = 1;
                        atomicOr(err, ERR_MAIN_PRODUCER);
                        ok = false;
                        break;
                    }
                    const int kk = back ? num_kb - 1 - kb : kb;
                    if (hook == 1 && leader && t == pair && kb == 0) {
                        // test hook: the leader never arms this stage, so the
                        // MMA thread's bounded wait on it runs out
                        if (++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * stage_bytes);
                    const uint32_t fb = full0 + 8u * static_cast<uint32_t>(s);
                    const uint32_t sa = base + s * STAGE;
                    // the k-block's A atoms, and the CTA's B column blocks, in
                    // one copy each when the sizes are whole blocks
                    if (chunked & 2) {
                        tma_load_4d_pair_hint(sa, &tmA, fb, 0, row, kk * KA, za, pol_a);
                    } else {
#pragma unroll
                        for (int j = 0; j < KA; ++j)
                            tma_load_3d_pair_hint(sa + j * A_ATOM, &tmA, fb, kk * BK + j * KG::AE,
                                                  row, za, pol_a);
                    }
                    if ((chunked & 1) && nbox > 1) {
                        tma_load_4d_pair_hint(sa + A_STAGE, &tmB4, fb, 0, kk * BK, col / KG::NB, zb,
                                              pol_b);
                    } else {
                        for (int j = 0; j < nbox; ++j)
                            tma_load_3d_pair_hint(sa + A_STAGE + j * KG::B_BOX, &tmB, fb,
                                                  col + j * KG::NB, kk * BK, zb, pol_b);
                    }
                    ++issued;
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Copies of both CTAs complete on the leader's full barriers, so the
            // leader waits there for the last min(issued, stages) armed phases;
            // the closing cluster barrier keeps the peer resident meanwhile.
            if (leader) {
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
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (leader only)
        if (leader && lane == 0) {
            constexpr uint32_t idesc_full = idesc_f16_f32(PM, PN, false, true);
            constexpr uint32_t idesc_half = idesc_f16_f32(PM, PN / 2, false, true);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                int b, tm, tn, half;
                work_item<ES>(t, tiles_m, tiles_n, group_m, whole, split_tail, b, tm, tn, half);
                const uint32_t idesc = half < 0 ? idesc_full : idesc_half;
                if (!mbar_wait(smem_u32(&tempty_bar[acc]), aph ^ 1u, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * PN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * STAGE;
                    // A: K-major, atoms of [128 rows][128 B of k] 16 KB apart, 8-row
                    // groups 1024 B apart, +32 B per MMA inside an atom.  B:
                    // MN-major, [BK k][128 B of n] boxes B_BOX apart, 8-row k
                    // groups 1024 B apart, one MMA's k rows per step.
                    const uint64_t ad = sdesc_sw128(sa, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sa + A_STAGE, KG::B_BOX, 1024);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        umma_pair<ES>(d, ad + ((k / 4) * (A_ATOM >> 4) + (k % 4) * 2),
                                      bd + KG::B_KSTEP * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(smem_u32(&empty_bar[s]), 0x3);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(smem_u32(&tfull_bar[acc]), 0x3);
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_MAIN_MMA);
            }
            umma_commit_pair(smem_u32(&drain_bar));
            if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;                       // TMEM lane quadrant of this warp
        const int wcol = (warp - 2) >> 2;             // which share of the columns
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty_bar[0]), 0);  // leader's
        const uint32_t stage_c = base + static_cast<uint32_t>(stages) * STAGE +
                                 static_cast<uint32_t>(warp - 2) * kStageC;
        int acc = 0;
        uint32_t aph = 0;
        for (int t = pair; t < total; t += npairs) {
            int b, tm, tn, half;
            work_item<ES>(t, tiles_m, tiles_n, group_m, whole, split_tail, b, tm, tn, half);
            void* Cb = batch_ptr(C, b, bt.sC, OUT_F32 ? 4 : 2);
            // a half item's accumulator has 128 columns, for output columns
            // from tn * 256 + half * 128
            const int span = half < 0 ? EPI_SPAN : EPI_SPAN / 2;
            const int c_lo = wcol * span;
            const int n0 = tn * PN + (half < 0 ? 0 : half * HN);
            const bool got = mbar_wait(smem_u32(&tfull_bar[acc]), aph, &abort_flag, epi_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    abort_flag = 1;
                    atomicOr(err, ERR_MAIN_EPILOGUE);
                }
                break;
            }
            tc_fence_after();
            const int m0 = tm * PM + static_cast<int>(rank) * HM + q * 32;  // this warp's first row
            const int m = m0 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * PN);
            // columns per TMA store: one 128-byte row of the box
            constexpr int G = OUT_F32 ? 32 : 64;
            if (c_tma) {
#pragma unroll 1
                for (int c = c_lo; c < c_lo + span; c += G) {
                    uint32_t r[G];
                    tmem_ld_32x32b_x32(taddr + c, *reinterpret_cast<uint32_t(*)[32]>(r));
                    if constexpr (G == 64)
                        tmem_ld_32x32b_x32(taddr + c + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                    tmem_ld_wait();
                    const int n = n0 + c;
                    if (m0 < M && n < N) {  // warp-uniform
                        if (epi.on && m < M) {
#pragma unroll
                            for (int j = 0; j < G; j += 32)
                                epilogue_chunk<OUT_F32>(r + j, m, n + j, N, epi);
                        }
                        // the staging buffer is free once the previous store
                        // has read it
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                        stage_store_box<OUT_F32>(&tmC, stage_c, r, n, m0, b, lane);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = c_lo; c < c_lo + span; c += EPI_COLS) {
                    uint32_t r[EPI_COLS];
                    if constexpr (EPI_COLS == 128) tmem_ld_32x32b_x128(taddr + c, r);
                    else if constexpr (EPI_COLS == 64) tmem_ld_32x32b_x64(taddr + c, r);
                    else tmem_ld_32x32b_x32(taddr + c, *reinterpret_cast<uint32_t(*)[32]>(r));
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < EPI_COLS; j += 32) {
                        const int n = n0 + c + j;
                        if (m < M && n < N) {
                            if (epi.on) epilogue_chunk<OUT_F32>(r + j, m, n, N, epi);
                            store_chunk<OUT_F32>(Cb, ldc, m, n, N, r + j, c_vec != 0);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_cluster(tempty0 + 8u * static_cast<uint32_t>(acc));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        // the TMA stores have read their staging buffers before the CTA
        // ends (their writes to C complete with the grid)
        if (c_tma && lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }

    pdl_trigger();  // this CTA has issued all its global writes
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

std::mutex g_mu;
bool g_attr_set[64][4];
int g_max_clusters[64][4];

template <bool OUT_F32, int ES>
cudaError_t launch_cfg(const GemmArgs& a)
{
    using KG = PairK<ES>;
    auto kernel = gemm_tc_pair_kernel<OUT_F32, ES>;
    const int slot = (OUT_F32 ? 1 : 0) + (ES == 1 ? 2 : 0);
    int max_clusters = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_attr_set[dev][slot]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(SMEM + kStageCBytes));
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2 * a.num_sms);
            q.blockDim = dim3(kThreads);
            q.dynamicSmemBytes = SMEM + kStageCBytes;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            q.attrs = at;
            q.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
            if (e != cudaSuccess) return e;
            g_max_clusters[dev][slot] = n > 0 ? n : 1;
            g_attr_set[dev][slot] = true;
        }
        max_clusters = g_max_clusters[dev][slot];
    }
    // A's KA atoms of a k-block in one copy when K is a whole number of
    // atoms (bit 1), and a CTA's HN / NB column blocks of B in one copy when
    // N is a whole number of blocks (bit 0, through a second map: the halves
    // of a cut last wave load one block through the first)
    CUtensorMap ta, tb, tb4;
    std::memset(&tb4, 0, sizeof(tb4));
    const int chunk_a = a.K % KG::AE == 0 ? 2 : 0;
    const int chunk_b = HN > KG::NB && a.N % KG::NB == 0 ? 1 : 0;
    if (chunk_a ? !encode_tmap_chunks(&ta, a.A, ES, static_cast<uint64_t>(a.K),
                                      static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda),
                                      a.batch, a.sA, KG::AE, HM, KA)
                : !encode_tmap(&ta, a.A, ES, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                               static_cast<uint64_t>(a.lda), a.batch, a.sA, KG::AE, HM))
        return cudaErrorInvalidValue;
    if (!encode_tmap(&tb, a.B, ES, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                     static_cast<uint64_t>(a.ldb), a.batch, a.sB, KG::NB, KG::BK))
        return cudaErrorInvalidValue;
    if (chunk_b &&
        !encode_tmap_chunks(&tb4, a.B, ES, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                            static_cast<uint64_t>(a.ldb), a.batch, a.sB, KG::NB, KG::BK,
                            HN / KG::NB))
        return cudaErrorInvalidValue;
    const int chunked = chunk_a | chunk_b;
    const int tiles_m = (a.M + PM - 1) / PM;
    const int tiles_n = (a.N + PN - 1) / PN;
    const int total = tiles_m * tiles_n * a.batch;
    const int split_tail = ES == 2 ? pair_split_tail(total, max_clusters, a.split_tail) : 0;
    const int items = total + split_tail;
    const int pairs = items < max_clusters ? items : max_clusters;
    const int group_m = a.group_m > 0 ? a.group_m : 8;
    const size_t es = OUT_F32 ? 4 : 2;
    const int c_vec = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) &&
                      ((static_cast<size_t>(a.ldc) * es) % 16 == 0) &&
                      ((static_cast<size_t>(a.sC) * es) % 16 == 0);
    // C written by TMA stores when the TMA engine can address it and its
    // rows end on a 16-byte boundary (at the right edge a TMA store writes
    // whole 16-byte units; columns N..ldc-1 stay untouched)
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    const int c_tma = c_vec && (static_cast<size_t>(a.N) * es) % 16 == 0 &&
                      encode_tmap_store(&tc, a.C, static_cast<int>(es),
                                        static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M),
                                        static_cast<uint64_t>(a.ldc), a.batch, a.sC,
                                        static_cast<uint32_t>(128 / es), 32);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    const int stages = a.stages > 0 ? a.stages : STAGES;
    if (stages < 2 || stages > STAGES) return cudaErrorInvalidValue;
    cfg.dynamicSmemBytes = stages * STAGE + (c_tma ? kStageCBytes : 0u) + 1024;
    cfg.stream = a.stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    set_pdl_attr(at[1]);
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tb4, tc, a.C, a.ldc, a.M, a.N, a.K, tiles_m,
                              tiles_n, group_m, split_tail, stages, c_vec, c_tma, chunked, a.hook,
                              a.err, a.epi, a.batch_args());
}

}  // namespace

int pair_split_tail(int total, int max_pairs, int forced)
{
    if (total <= 0 || max_pairs <= 0) return 0;
    if (forced >= 0) return forced < total ? forced : total;
    // Tiles go to the pairs in waves of max_pairs.  The last wave holds
    // `last` tiles; when twice that many fit in one wave, each of them is
    // cut into two 256 x 128 halves.  An M = 256, N = 128 pair MMA costs
    // ~98 cycles against ~128 for N = 256 (measured), so the wave then takes
    // ~0.77 of a whole-tile wave, on twice as many pairs.
    const int last = total - max_pairs * ((total - 1) / max_pairs);
    return 2 * last <= max_pairs ? last : 0;
}

int pair_max_stages() { return STAGES; }

int pair_tiles(int M, int N)
{
    return ((M + PM - 1) / PM) * ((N + PN - 1) / PN);
}

cudaError_t launch_main_pair(const GemmArgs& a)
{
    if (a.in_es == 1) return a.out_f32 ? launch_cfg<true, 1>(a) : launch_cfg<false, 1>(a);
    return a.out_f32 ? launch_cfg<true, 2>(a) : launch_cfg<false, 2>(a);
}

}  // namespace tg

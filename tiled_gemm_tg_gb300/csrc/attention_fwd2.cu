// attention_fwd2.cu -- attention forward O = softmax(scale * Q K^T) V for heads
// with d <= 128 and dv <= 128, the probabilities kept in tensor memory.
//
// The operation and its blockwise evaluation are those of "TileLang实战：用
// Python DSL自动生成高性能GPU计算内核" (gsyq.cn), §4 (FlashAttention): keys and
// values are consumed in blocks, each query row keeps its running maximum M
// and normaliser L, and the output is rescaled when M grows.  The general
// kernel (attention_fwd.cu) computes the same thing for any d and dv; this
// one is laid out for the common head sizes.
//
// GB300 design.  A CTA owns 128 query rows and walks the keys in blocks of
// 128, with two TMEM score buffers b = t % 2:
//   S_t = Q K_t^T      tcgen05.mma M=128 N=128, K = d (Q resident, the key
//                      block one TMA stage), into TMEM columns 128b..128b+127;
//   P_t = exp2(S_t * scale * log2 e - m)   two threads per query row (64
//                      scores each, one tcgen05.ld) agree on the row maximum
//                      and write P as fp16 pairs over the first 64 of those
//                      columns;
//   [O | L] += P_t [V_t | 1]   tcgen05.mma M=128 N=144 with A = P_t from
//                      TMEM, B = V_t from shared memory (MN-major) followed
//                      by a box of ones, accumulating in TMEM columns 256 ..
//                      399: columns 128.. of the product are the normaliser
//                      L = sum_k p_k of exactly the fp16 weights the MMA
//                      used, so the softmax threads never sum P themselves.
// S_(t+1) goes to the other buffer, so the tensor core computes it while the
// softmax turns S_t into P_t; S_(t+2) reuses buffer b once P_t V_t has
// completed.  P never leaves tensor memory: no shared-memory round trip and
// no proxy fence between the softmax and the MMA.  Each tcgen05.commit ends
// a whole block of MMAs: a commit after a few MMAs leaves the pipe idle.
// The running maximum is raised only when a block's maximum exceeds it by
// more than 8 (base 2); then the row of [O | L] (in TMEM) is scaled by
// 2^(m_old - m_new) before P_t V_t is issued.
//
// Warp roles (384 threads): 0 TMA for Q (once) and K, 1 TMEM allocation and
// the S MMAs, 2 TMA for V, 3 the P V MMAs, 4-11 softmax and output (warp w
// reads TMEM lane quadrant w % 4; two warps per quadrant split the keys).
// Every wait is bounded: on expiry a role records it in the device error
// word, raises the CTA's abort flag and winds down.
//
// The grid is one CTA per tile (128 query rows of one batch entry), issued
// in waves of one tile per SM.  Given a workspace, the tiles of a short last
// wave are each cut into 2 or 4 consecutive ranges of key blocks, one CTA
// per range (attention_tail_plan says which): a range writes its
// unnormalised O, maximum and normaliser to the workspace, counts itself on
// the tile's counter, and the range that counts last merges all of them in
// range order, the same merge the blockwise pass applies between blocks.  A
// one-CTA kernel zeroes the counters first.  The dispatcher hands the short
// ranges to SMs as they free up, so the SMs finish closer together.
#include <cstdint>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

using namespace tg::dev;

constexpr int BM = 128;                        // query rows per CTA
constexpr int BN = 128;                        // keys per block
constexpr int DC = 64;                         // d per chunk: 128 bytes of fp16
constexpr int QC = 2;                          // Q chunks (d <= 128)
constexpr uint32_t Q_CHUNK = BM * DC * 2;      // 16 KB
constexpr uint32_t K_CHUNK = BN * DC * 2;      // 16 KB
constexpr uint32_t K_BLK = QC * K_CHUNK;       // a key block: one stage, one release
constexpr uint32_t V_BOX = BN * 128;           // [128 keys][64 columns] fp16, 16 KB
// a V stage: two boxes of V (128 output columns) and a box of ones, so that
// the P V MMA's columns 128.. accumulate the normaliser sum_k p_k
constexpr uint32_t V_STAGE = 3 * V_BOX;
constexpr uint32_t Q_RES = QC * Q_CHUNK;       // 32 KB
constexpr int V_STAGES = 2;
// 227 KB per CTA covers static shared memory too (barriers and the row
// exchange array, about 2.2 KB): keep 8 KB for it
constexpr uint32_t BUDGET = 227 * 1024 - 8192;
constexpr int K_STAGES =
    static_cast<int>((BUDGET - 1024 - Q_RES - V_STAGES * V_STAGE) / K_BLK);
constexpr uint32_t SMEM = 1024 + Q_RES + V_STAGES * V_STAGE + K_STAGES * K_BLK;
static_assert(K_STAGES >= 2, "too few key stages");
static_assert(SMEM <= BUDGET, "shared-memory budget exceeded");
constexpr int NBUF = 2;                        // TMEM score buffers
constexpr uint32_t TMEM_COLS = 512;            // S/P buffers 0 and 1, then O
constexpr uint32_t O_COL = NBUF * BN;
constexpr int O_N = 144;                       // O: 128 output columns, then the normaliser
static_assert(O_COL + O_N <= TMEM_COLS, "tensor memory exceeded");
constexpr int kThreads = 384;                  // 4 role warps + 8 softmax warps
constexpr int HK = BN / 2;                     // keys per softmax warp
constexpr float kRescaleLog2 = 8.0f;
// Tail split: the tiles of a last wave that holds at most kTailFill4
// percent of the SMs' worth of tiles are cut into 4 pieces along the keys,
// of at most kTailFill2 percent into 2, each piece at least kTailMinBlocks
// key blocks.
constexpr int kMaxPieces = 4;
constexpr int kTailFill4 = 20;
constexpr int kTailFill2 = 45;
constexpr int kTailMinBlocks = 4;

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
attention_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, void* O, long long ldo, long long sO,
                      int Nq, int Nk, int dv, int n_chunks, float scale_log2, int o_vec, int zq,
                      int zk, int zv, int q_blocks, int units_full, int pieces, float* tws_o, float* tws_ml,
                      unsigned int* tws_cnt, int hook, unsigned int* err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t k_full[K_STAGES];
    __shared__ __align__(8) uint64_t k_empty[K_STAGES];
    __shared__ __align__(8) uint64_t q_full;
    __shared__ __align__(8) uint64_t v_full[V_STAGES];
    __shared__ __align__(8) uint64_t v_empty[V_STAGES];
    __shared__ __align__(8) uint64_t s_full[NBUF]; // S of the buffer's block is in TMEM
    __shared__ __align__(8) uint64_t p_full[NBUF]; // P written over it (256 arrivals)
    __shared__ __align__(8) uint64_t pv_done[NBUF];  // the buffer's P V MMAs are complete
    __shared__ __align__(8) uint64_t drain_s;
    __shared__ __align__(8) uint64_t drain_o;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ unsigned int tail_old;
    __shared__ float red[NBUF][2][BM];  // per-row partial maxima of the two halves, by buffer

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t q_res = base;
    const uint32_t k_base = base + Q_RES;
    const uint32_t v_base = k_base + K_STAGES * K_BLK;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work units: units 0 .. units_full-1 are whole tiles (128 query rows of
    // one batch entry, all keys); each tile after them, a tile of the last,
    // partial wave, is cut into `pieces` consecutive ranges of key blocks,
    // one unit per range, merged by whichever unit of the tile ends last.
    const int unit = static_cast<int>(blockIdx.x);
    int tile = unit;
    int part = -1;
    if (unit >= units_full) {
        tile = units_full + (unit - units_full) / pieces;
        part = (unit - units_full) % pieces;
    }
    const int q0 = (tile % q_blocks) * BM;
    const int bz = tile / q_blocks;
    const int n_kv_all = (Nk + BN - 1) / BN;
    const int kv0 = part < 0 ? 0 : part * n_kv_all / pieces;
    const int n_kv = (part < 0 ? n_kv_all : (part + 1) * n_kv_all / pieces) - kv0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < K_STAGES; ++s) {
            mbar_init(smem_u32(&k_full[s]), 1);
            mbar_init(smem_u32(&k_empty[s]), 1);
        }
        for (int s = 0; s < V_STAGES; ++s) {
            mbar_init(smem_u32(&v_full[s]), 1);
            mbar_init(smem_u32(&v_empty[s]), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(smem_u32(&s_full[b]), 1);
            mbar_init(smem_u32(&p_full[b]), 2 * BM);
            mbar_init(smem_u32(&pv_done[b]), 1);
        }
        mbar_init(smem_u32(&q_full), 1);
        mbar_init(smem_u32(&drain_s), 1);
        mbar_init(smem_u32(&drain_o), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // the third box of every V stage holds ones (fp16 1.0): TMA never writes it
    for (int i = threadIdx.x; i < V_STAGES * static_cast<int>(V_BOX / 16); i += kThreads) {
        const int st = i / static_cast<int>(V_BOX / 16);
        const int j = i - st * static_cast<int>(V_BOX / 16);
        st_shared_v4(v_base + st * V_STAGE + 2 * V_BOX + 16u * j, 0x3c003c00u, 0x3c003c00u, 0x3c003c00u,
                     0x3c003c00u);
    }
    fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    // a softmax step waits for a whole block of MMAs; allow ~64 us per chunk
    const uint32_t long_limit =
        kSlowPolls + 64u * static_cast<uint32_t>(min(n_chunks + 8, 1 << 20));

    if (warp == 0) {
        // --------------------------------------------------- TMA: Q and K
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0;
            const uint32_t qb = smem_u32(&q_full);
            mbar_arrive_expect_tx(qb, static_cast<uint32_t>(n_chunks) * Q_CHUNK);
            for (int c = 0; c < n_chunks; ++c)
                tma_load_3d(q_res + c * Q_CHUNK, &tmQ, qb, c * DC, q0, bz * zq);
            for (int t = 0; t < n_kv; ++t) {
                if (!mbar_wait(smem_u32(&k_empty[s]), ph ^ 1u, &abort_flag, long_limit)) {
                    abort_flag = 1;
                    atomicOr(err, ERR_ATTENTION);
                    break;
                }
                if (!(hook == 1 && t == 0)) {  // test hook: leave the first stage empty
                    const uint32_t fb = smem_u32(&k_full[s]);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(n_chunks) * K_CHUNK);
                    for (int c = 0; c < n_chunks; ++c)
                        tma_load_3d(k_base + s * K_BLK + c * K_CHUNK, &tmK, fb, c * DC, (kv0 + t) * BN,
                                    bz * zk);
                    ++issued;
                }
                if (++s == K_STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // wait for this thread's copies still in flight before leaving
            for (uint32_t i = 0; i < min(issued, static_cast<uint32_t>(K_STAGES)); ++i) {
                if (--s < 0) {
                    s = K_STAGES - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&k_full[s]), ph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
            if (!mbar_wait(qb, 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------- TMA: V
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0;
            for (int t = 0; t < n_kv; ++t) {
                if (!mbar_wait(smem_u32(&v_empty[s]), ph ^ 1u, &abort_flag, long_limit)) {
                    abort_flag = 1;
                    atomicOr(err, ERR_ATTENTION);
                    break;
                }
                const uint32_t fb = smem_u32(&v_full[s]);
                const uint32_t sv = v_base + s * V_STAGE;
                mbar_arrive_expect_tx(fb, 2 * V_BOX);  // the two V boxes (the third is ones)
                tma_load_3d(sv, &tmV, fb, 0, (kv0 + t) * BN, bz * zv);
                tma_load_3d(sv + V_BOX, &tmV, fb, 64, (kv0 + t) * BN, bz * zv);
                ++issued;
                if (++s == V_STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            for (uint32_t i = 0; i < min(issued, static_cast<uint32_t>(V_STAGES)); ++i) {
                if (--s < 0) {
                    s = V_STAGES - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&v_full[s]), ph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------ MMA issuer: S = Q K^T
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(BM, BN, false, false);
            int ks = 0;
            uint32_t kph = 0;
            bool ok = mbar_wait(smem_u32(&q_full), 0, &abort_flag);
            for (int t = 0; t < n_kv && ok; ++t) {
                const int b = t % NBUF;
                // buffer b held P_(t-NBUF): reuse it once that block's P V has completed
                if (t >= NBUF && !mbar_wait(smem_u32(&pv_done[b]), static_cast<uint32_t>((t / NBUF - 1) & 1),
                                            &abort_flag, long_limit)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(smem_u32(&k_full[ks]), kph, &abort_flag, long_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_s = tmem_base + static_cast<uint32_t>(b * BN);
                for (int c = 0; c < n_chunks; ++c) {
                    // both operands K-major: 8-row groups 1024 B apart, +32 B per 16 of d
                    const uint64_t ad = sdesc_sw128(q_res + c * Q_CHUNK, 16, 1024);
                    const uint64_t bd = sdesc_sw128(k_base + ks * K_BLK + c * K_CHUNK, 16, 1024);
#pragma unroll
                    for (int k = 0; k < DC / 16; ++k)
                        umma_f16(d_s, ad + 2ull * k, bd + 2ull * k, idesc_s, (c | k) != 0 ? 1u : 0u);
                }
                umma_commit(smem_u32(&s_full[b]));
                umma_commit(smem_u32(&k_empty[ks]));
                if (++ks == K_STAGES) {
                    ks = 0;
                    kph ^= 1u;
                }
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
            // every MMA this thread issued must finish before TMEM is freed
            umma_commit(smem_u32(&drain_s));
            if (!mbar_wait(smem_u32(&drain_s), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------ MMA issuer: O += P V
        if (lane == 0) {
            // A = P from TMEM (K-major), B = V from shared memory (MN-major)
            constexpr uint32_t idesc_o = idesc_f16_f32(BM, O_N, false, true);
            int vs = 0;
            uint32_t vph = 0;
            bool ok = true;
            for (int t = 0; t < n_kv; ++t) {
                const int b = t % NBUF;
                if (!mbar_wait(smem_u32(&p_full[b]), static_cast<uint32_t>((t / NBUF) & 1), &abort_flag,
                               long_limit) ||
                    !mbar_wait(smem_u32(&v_full[vs]), vph, &abort_flag, long_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // V: 64-column boxes 16 KB apart (the third one ones), 16 keys =
                // 2048 B per step
                const uint64_t bd = sdesc_sw128(v_base + vs * V_STAGE, V_BOX, 1024);
                const uint32_t a_tm = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    umma_f16_ts(tmem_base + O_COL, a_tm + 8u * k, bd + 128ull * k, idesc_o,
                                (t | k) != 0 ? 1u : 0u);
                umma_commit(smem_u32(&pv_done[b]));
                umma_commit(smem_u32(&v_empty[vs]));
                if (++vs == V_STAGES) {
                    vs = 0;
                    vph ^= 1u;
                }
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
            umma_commit(smem_u32(&drain_o));
            if (!mbar_wait(smem_u32(&drain_o), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax and output
        // Two warps per TMEM lane quadrant: warp h of the pair takes keys
        // h*64 .. h*64+63 of each block (and output columns h*64 ..); the
        // pair agrees on each row's maximum through shared memory and a
        // 64-thread named barrier.  The row's sum comes from the MMA.
        const int qd = warp & 3;          // TMEM lane quadrant
        const int h = (warp - 4) >> 2;    // which half of the keys
        const int r = qd * 32 + lane;     // this thread's query row
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
        const bool pos_scale = scale_log2 >= 0.0f;
        float m_run = -INFINITY;          // running maximum, base-2 scaled logits
        bool ok = true;
        // Every iteration passes exactly one pair barrier, also after a
        // failed wait (the work is then skipped), so the two warps of a pair
        // always meet; a failure raises the abort flag at once so that every
        // other role's bounded waits end too.
        auto fail = [&]() {
            ok = false;
            if (lane == 0) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
        };
        for (int t = 0; t < n_kv; ++t) {
            const int b = t % NBUF;
            const uint32_t s_col = static_cast<uint32_t>(b * BN);
            uint32_t raw[HK];
            float mine = 0.0f;
            const int valid = min(BN, Nk - (kv0 + t) * BN) - h * HK;
            if (ok) {
                const bool got = mbar_wait(smem_u32(&s_full[b]), static_cast<uint32_t>((t / NBUF) & 1),
                                           &abort_flag, long_limit);
                if (!__all_sync(0xffffffffu, got)) fail();
            }
            if (ok) {
                tc_fence_after();
                tmem_ld_32x32b_x64(t_lane + s_col + static_cast<uint32_t>(h * HK), raw);
                tmem_ld_wait();
                // keys past Nk (zero-filled by TMA) are masked; only the last
                // block can have them
                if (valid < HK) {
#pragma unroll
                    for (int j = 0; j < HK; ++j)
                        if (j >= valid) raw[j] = __float_as_uint(pos_scale ? -INFINITY : INFINITY);
                }
                // the extreme raw score of this half, in four chains
                float mc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) mc[c] = __uint_as_float(raw[c]);
                if (pos_scale) {
#pragma unroll
                    for (int j = 4; j < HK; ++j) mc[j & 3] = fmaxf(mc[j & 3], __uint_as_float(raw[j]));
                } else {
#pragma unroll
                    for (int j = 4; j < HK; ++j) mc[j & 3] = fminf(mc[j & 3], __uint_as_float(raw[j]));
                }
                mine = pos_scale ? fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]))
                                 : fminf(fminf(mc[0], mc[1]), fminf(mc[2], mc[3]));
            }
            // the exchange also orders both halves' score loads before either
            // half writes P over the buffer's first 64 columns
            red[b][h][r] = mine;
            named_bar_sync(1 + qd, 64);
            const float other = red[b][h ^ 1][r];
            if (!ok) continue;

            const float mraw = pos_scale ? fmaxf(mine, other) : fminf(mine, other);
            const float mx = mraw * scale_log2;
            const bool raise = mx > m_run + kRescaleLog2;
            float alpha = 1.0f;
            if (raise) {
                alpha = ex2_approx(m_run - mx);  // 0 for the first block
                m_run = mx;
            }
            const float neg_m = -m_run;

            // P = 2^(s * scale * log2 e - m) as fp16 pairs: this half's 64
            // keys go to columns h*32 .. h*32+31 of the buffer
            uint32_t pw[HK / 2];
            auto make_p = [&](auto masked) {
#pragma unroll
                for (int j = 0; j < HK; j += 2) {
                    float a0 = fmaf(__uint_as_float(raw[j]), scale_log2, neg_m);
                    float a1 = fmaf(__uint_as_float(raw[j + 1]), scale_log2, neg_m);
                    if constexpr (decltype(masked)::value) {
                        if (j >= valid) a0 = -INFINITY;
                        if (j + 1 >= valid) a1 = -INFINITY;
                    }
                    const __half2 v2 = __floats2half2_rn(ex2_approx(a0), ex2_approx(a1));
                    pw[j / 2] = *reinterpret_cast<const uint32_t*>(&v2);
                }
            };
            if (valid < HK) make_p(std::true_type{});
            else make_p(std::false_type{});
            tmem_st_32x32b_x32(t_lane + s_col + static_cast<uint32_t>(h * (HK / 2)), pw);
            if (t > 0 && __any_sync(0xffffffffu, raise)) {
                // then this half of O *= alpha (1 in rows that kept their
                // maximum), once P_(t-1) V has completed; P_t V waits for
                // this block's P
                const int u = t - 1;
                const bool got_o = mbar_wait(smem_u32(&pv_done[u % NBUF]), static_cast<uint32_t>((u / NBUF) & 1),
                                             &abort_flag, long_limit);
                if (!__all_sync(0xffffffffu, got_o)) {
                    tmem_st_wait();
                    fail();
                    continue;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < HK; c += 32) {
                    const uint32_t col = O_COL + static_cast<uint32_t>(h * HK + c);
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(t_lane + col, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st_32x32b_x32(t_lane + col, o);
                }
                if (h == 1) {
                    // the normaliser columns
                    uint32_t o[16];
                    tmem_ld_32x32b_x16(t_lane + O_COL + 128u, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st_32x32b_x16(t_lane + O_COL + 128u, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&p_full[b]));
        }
        if (ok && n_kv > 0) {
            // the last block's MMAs complete O
            const int u = n_kv - 1;
            const bool got = mbar_wait(smem_u32(&pv_done[u % NBUF]), static_cast<uint32_t>((u / NBUF) & 1),
                                       &abort_flag, long_limit);
            if (!__all_sync(0xffffffffu, got)) fail();
        }
        if (ok) {
            tc_fence_after();
        }
        const int m = q0 + r;
        void* Ob = batch_ptr(O, bz, sO, OUT_F32 ? 4 : 2);
        if (part < 0) {
            if (ok) {
                // the row's normaliser: column 128 of O, the weights (the
                // fp16 ones the MMA used) summed by the P V MMA against the ones
                uint32_t lw[16];
                tmem_ld_32x32b_x16(t_lane + O_COL + 128u, lw);
                tmem_ld_wait();
                const float inv_l = 1.0f / __uint_as_float(lw[0]);
#pragma unroll 1
                for (int c = 0; c < HK; c += 32) {
                    const int n = h * HK + c;
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(n), o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv_l);
                    if (m < Nq && n < dv) store_chunk<OUT_F32>(Ob, ldo, m, n, dv, o, o_vec != 0);
                }
            }
        } else {
            // One piece of a tail tile: its unnormalised O, running maximum
            // and normaliser go to the workspace; the piece that ends last
            // merges them all, O = sum_p w_p O_p / sum_p w_p L_p with
            // w_p = 2^(m_p - max_p m_p), in the order of the pieces whichever
            // unit merges, so that every call rounds alike.  A piece's O is
            // stored column by column (128 rows of a column contiguous), so
            // that a warp's 32 rows make one 128-byte line per access.
            const int ti = tile - units_full;
            const size_t slot0 = static_cast<size_t>(ti) * pieces;  // piece p: slot0 + p
            const size_t slot_self = slot0 + static_cast<size_t>(part);
            if (ok) {
                uint32_t lw[16];
                tmem_ld_32x32b_x16(t_lane + O_COL + 128u, lw);
                tmem_ld_wait();
#pragma unroll 1
                for (int c = 0; c < HK; c += 32) {
                    const int n = h * HK + c;
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(n), o);
                    tmem_ld_wait();
                    float* dst = tws_o + (slot_self * 128 + static_cast<size_t>(n)) * BM + r;
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[static_cast<size_t>(e) * BM] = __uint_as_float(o[e]);
                }
                if (h == 0) {
                    tws_ml[2 * (slot_self * BM + r)] = m_run;
                    tws_ml[2 * (slot_self * BM + r) + 1] = __uint_as_float(lw[0]);
                }
            }
            __threadfence();  // this thread's partial is visible before the count
            named_bar_sync(5, 2 * BM);
            if (warp == 4 && lane == 0) {
                pdl_wait();  // the counters were zeroed by the kernel before this one
                tail_old = abort_flag == 0 ? atomicAdd(&tws_cnt[ti], 1u) : 0xffffffffu;
            }
            named_bar_sync(5, 2 * BM);
            if (ok && tail_old == static_cast<unsigned int>(pieces - 1)) {
                __threadfence();  // the other pieces, counted before this one, are visible
                // read through L2: the other pieces' lines were written by other SMs
                const float* ml = tws_ml + 2 * (slot0 * BM + r);  // piece p: ml[2 * p * BM]
                float mm = -INFINITY;
#pragma unroll 1
                for (int p = 0; p < pieces; ++p) mm = fmaxf(mm, __ldcg(ml + 2 * p * BM));
                float lsum = 0.0f;
#pragma unroll 1
                for (int p = 0; p < pieces; ++p)
                    lsum = fmaf(ex2_approx(__ldcg(ml + 2 * p * BM) - mm), __ldcg(ml + 2 * p * BM + 1), lsum);
                const float inv = 1.0f / lsum;
#pragma unroll 1
                for (int c = 0; c < HK; c += 32) {
                    const int n = h * HK + c;
                    float acc[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
                    // two pieces' columns in flight at a time (pieces >= 2)
#pragma unroll 1
                    for (int p = 0; p < pieces; p += 2) {
                        const int p1 = p + 1 < pieces ? p + 1 : p;
                        const float w0 = ex2_approx(__ldcg(ml + 2 * p * BM) - mm);
                        const float w1 = p1 != p ? ex2_approx(__ldcg(ml + 2 * p1 * BM) - mm) : 0.0f;
                        const float* s0 = tws_o + ((slot0 + p) * 128 + static_cast<size_t>(n)) * BM + r;
                        const float* s1 = tws_o + ((slot0 + p1) * 128 + static_cast<size_t>(n)) * BM + r;
                        float v0[32], v1[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            v0[e] = __ldcg(s0 + static_cast<size_t>(e) * BM);
                            v1[e] = __ldcg(s1 + static_cast<size_t>(e) * BM);
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = fmaf(w1, v1[e], fmaf(w0, v0[e], acc[e]));
                    }
                    uint32_t o[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(acc[e] * inv);
                    if (m < Nq && n < dv) store_chunk<OUT_F32>(Ob, ldo, m, n, dv, o, o_vec != 0);
                }
                if (warp == 4 && lane == 0) tws_cnt[ti] = 0u;  // ready for the next call
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Zeroes the tail tiles' counters; lets the attention kernel, launched as
// its programmatic dependent, start at once (only the tail units wait for
// this grid, just before they count).
__global__ void __launch_bounds__(256) tail_zero_kernel(unsigned int* cnt, int n)
{
    pdl_trigger();
    for (int i = static_cast<int>(threadIdx.x); i < n; i += static_cast<int>(blockDim.x)) cnt[i] = 0u;
}

std::mutex g_attr_mu;
bool g_attr_set[64][2];

template <bool OUT_F32>
cudaError_t launch_cfg(const AttnArgs& a)
{
    auto kernel = attention_fwd2_kernel<OUT_F32>;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(g_attr_mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!g_attr_set[dev][OUT_F32 ? 1 : 0]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(SMEM));
            if (e != cudaSuccess) return e;
            g_attr_set[dev][OUT_F32 ? 1 : 0] = true;
        }
    }
    CUtensorMap tq, tk, tv;
    if (!encode_tmap(&tq, a.Q, 2, static_cast<uint64_t>(a.d), static_cast<uint64_t>(a.Nq),
                     static_cast<uint64_t>(a.ldq), a.batch, a.sQ, DC, BM) ||
        !encode_tmap(&tk, a.K, 2, static_cast<uint64_t>(a.d), static_cast<uint64_t>(a.Nk),
                     static_cast<uint64_t>(a.ldk), a.batch, a.sK, DC, BN) ||
        !encode_tmap(&tv, a.V, 2, static_cast<uint64_t>(a.dv), static_cast<uint64_t>(a.Nk),
                     static_cast<uint64_t>(a.ldv), a.batch, a.sV, 64, BN))
        return cudaErrorInvalidValue;
    const size_t es = OUT_F32 ? 4 : 2;
    const int o_vec = (reinterpret_cast<uintptr_t>(a.O) % 16 == 0) &&
                      ((static_cast<size_t>(a.ldo) * es) % 16 == 0) &&
                      ((static_cast<size_t>(a.sO) * es) % 16 == 0);
    const int q_blocks = (a.Nq + BM - 1) / BM;
    const long long tiles = static_cast<long long>(q_blocks) * a.batch;
    const int tail = a.tail_tiles;  // tiles of the last wave cut into pieces along the keys
    const int pieces = tail > 0 ? a.tail_pieces : 1;
    if (tail < 0 || tail > tiles || (tail > 0 && a.ws == nullptr) || pieces < 1 ||
        pieces > kMaxPieces || (tail > 0 && (pieces < 2 || pieces > (a.Nk + BN - 1) / BN)))
        return cudaErrorInvalidValue;
    const long long units = tiles - tail + static_cast<long long>(tail) * pieces;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(units), 1, 1);
    float* tws_o = nullptr;
    float* tws_ml = nullptr;
    unsigned int* tws_cnt = nullptr;
    if (tail > 0) {
        tws_o = static_cast<float*>(a.ws);
        tws_ml = tws_o + attention_tail_o_floats(tail, pieces);
        tws_cnt = reinterpret_cast<unsigned int*>(tws_ml + attention_tail_ml_floats(tail, pieces));
        tail_zero_kernel<<<1, 256, 0, a.stream>>>(tws_cnt, tail);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const float scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)
    const int n_chunks = (a.d + DC - 1) / DC;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = a.stream;
    cudaLaunchAttribute at[1];
    set_pdl_attr(at[0]);
    cfg.attrs = at;
    cfg.numAttrs = tail > 0 ? 1 : 0;  // only behind the counter-zeroing kernel
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, a.O, a.ldo, a.sO, a.Nq, a.Nk, a.dv, n_chunks,
                              scale_log2, o_vec, static_cast<int>(a.sQ != 0),
                              static_cast<int>(a.sK != 0), static_cast<int>(a.sV != 0), q_blocks,
                              static_cast<int>(tiles - tail), pieces, tws_o, tws_ml, tws_cnt, a.hook,
                              a.err);
}

}  // namespace

long long attention_tail_o_floats(int tail, int pieces)
{
    // fp32 [tail][pieces][128 columns][128 rows], 256-byte aligned after it
    return (static_cast<long long>(tail) * pieces * BM * 128 + 63) / 64 * 64;
}

long long attention_tail_ml_floats(int tail, int pieces)
{
    // fp32 [tail][pieces][128 rows][maximum, normaliser]
    return (static_cast<long long>(tail) * pieces * BM * 2 + 63) / 64 * 64;
}

int attention_tail_plan(int batch, int Nq, int Nk, int num_sms, int* pieces)
{
    // Tiles go to the SMs in waves.  When the tiles fill the SMs more than
    // once and the last wave is short, each tile of that wave is cut into
    // pieces along the keys; the dispatcher hands the short pieces to SMs as
    // they free up, so that the SMs end closer together.  Each piece costs
    // its own start (Q load, pipeline fill), a partial write, and a share of
    // the merge, which outweighs the gain once the last wave is about half
    // full: the thresholds are measured ones.
    *pieces = 0;
    if (batch <= 0 || Nq <= 0 || Nk <= 0 || num_sms <= 0) return 0;
    const long long tiles = static_cast<long long>((Nq + BM - 1) / BM) * batch;
    const int n_kv = (Nk + BN - 1) / BN;
    if (tiles <= num_sms) return 0;
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const long long tail = tiles - (waves - 1) * num_sms;
    int p = 0;
    if (tail * 100 <= static_cast<long long>(num_sms) * kTailFill4) p = 4;
    else if (tail * 100 <= static_cast<long long>(num_sms) * kTailFill2) p = 2;
    if (p > n_kv / kTailMinBlocks) p = n_kv / kTailMinBlocks;
    if (p > kMaxPieces) p = kMaxPieces;
    if (p < 2) return 0;
    *pieces = p;
    return static_cast<int>(tail);
}

size_t attention_tail_ws_bytes(int batch, int Nq, int Nk, int num_sms)
{
    int pieces = 0;
    const int tail = attention_tail_plan(batch, Nq, Nk, num_sms, &pieces);
    if (tail == 0) return 0;
    return static_cast<size_t>(attention_tail_o_floats(tail, pieces) +
                               attention_tail_ml_floats(tail, pieces)) *
               sizeof(float) +
           static_cast<size_t>(tail) * sizeof(unsigned int);
}

bool attention_tmem_p_serves(int d, int dv)
{
    return d >= 1 && d <= DC * QC && dv >= 1 && dv <= 128;
}

cudaError_t launch_attention_tmem_p(const AttnArgs& a)
{
    if (!attention_tmem_p_serves(a.d, a.dv) || a.Nk < 1) return cudaErrorInvalidValue;
    return a.out_f32 ? launch_cfg<true>(a) : launch_cfg<false>(a);
}

}  // namespace tg

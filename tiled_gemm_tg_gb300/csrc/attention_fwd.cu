// attention_fwd.cu -- attention forward O = softmax(scale * Q K^T) V on the
// tensor cores, one pass over the keys with a running maximum and normaliser.
//
// The operation and its blockwise evaluation are those of "TileLang实战：用
// Python DSL自动生成高性能GPU计算内核" (gsyq.cn), §4 (FlashAttention): keys and
// values are consumed in blocks, each query row keeps its running maximum M
// and normaliser L, and the output is rescaled when M grows, so the Nq x Nk
// score matrix never exists in memory.  The page's kernel uses no 1/sqrt(d)
// factor; `scale` is a parameter (1 reproduces it).
//
// GB300 design.  A CTA owns 128 query rows and a slice of DVS (128 or 256)
// output columns, and walks the keys in blocks of 128:
//   S_t = Q K_t^T      tcgen05.mma, M=128 N=128, K = d in 64-wide chunks
//                      (Q and K chunks streamed together by TMA), into one of
//                      two 128-column TMEM buffers;
//   P_t = exp2(S_t * scale * log2 e - m)   softmax warps, one query row per
//                      thread, fp16 P written to shared memory in the
//                      128-byte-swizzled K-major layout the MMA reads;
//   O += P_t V_t       tcgen05.mma, M=128 N=DVS K=128, V MN-major from TMA,
//                      accumulating in TMEM columns 256 .. 256+DVS.
// Two threads issue the MMAs: one the scores (up to two blocks ahead, into
// alternating S buffers), the other P_t V_t as soon as P_t is written, so
// the tensor core works on the next scores while the softmax warps turn S_t
// into P_t and neither stream waits behind the other's barriers.  The running
// maximum is raised only when a block's maximum exceeds it by more than 8 (in
// base 2): then O (in TMEM) and L are scaled by 2^(m_old - m_new); otherwise
// the stale maximum stays, the probabilities stay below 2^8, and the final
// O / L is the same quotient.  Outputs wider than 256 columns take several
// CTAs, each recomputing S for its own slice of V.
//
// Warp roles (384 threads): 0 TMA for Q and K, 1 TMEM allocation and the
// S MMAs, 2 TMA for V, 3 the P V MMAs, 4-11 softmax and output (warp w reads
// TMEM lane quadrant w % 4; two warps per quadrant split the keys).  Every wait is bounded: on expiry a role records it in
// the device error word, raises the CTA's abort flag and winds down.
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

constexpr int BM = 128;                       // query rows per CTA
constexpr int BN = 128;                       // keys per block
constexpr int DC = 64;                        // d per chunk: 128 bytes of fp16
constexpr uint32_t Q_CHUNK = BM * DC * 2;     // 16 KB
constexpr uint32_t K_CHUNK = BN * DC * 2;     // 16 KB
constexpr uint32_t P_ATOM = BM * 128;         // [128 rows][64 keys] fp16, 16 KB
constexpr uint32_t P_BUF = 2 * P_ATOM;        // 128 keys
constexpr uint32_t V_BOX = BN * 128;          // [128 keys][64 columns] fp16, 16 KB
constexpr uint32_t TMEM_COLS = 512;           // S0, S1 (128 each), O (<= 256)
constexpr uint32_t O_COL = 256;
constexpr int kThreads = 384;                 // 4 role warps + 8 softmax warps
constexpr uint32_t kSoftmaxThreads = 256;
constexpr float kRescaleLog2 = 8.0f;          // raise the running max past 2^8 growth

// QMODE: the number of 64-wide Q chunks kept resident in shared memory for
// the whole CTA (2: d <= 128, 4: d <= 256), so the ring carries K chunks
// only; or 0: Q is streamed with K, chunk by chunk, for any d.  The ring gets
// whatever shared memory the fixed parts leave.
template <int DVS, int QMODE>
struct AttnCfg {
    static_assert(DVS == 128 || DVS == 256, "an output slice is 128 or 256 columns");
    static_assert(QMODE == 0 || QMODE == 2 || QMODE == 4, "resident Q of 0, 2 or 4 chunks");
    static constexpr uint32_t V_STAGE = BN * DVS * 2;
    static constexpr uint32_t Q_RES = QMODE * Q_CHUNK;
    static constexpr uint32_t STAGE = QMODE ? K_CHUNK : Q_CHUNK + K_CHUNK;
    // 227 KB per CTA covers static shared memory too: keep 4 KB for it
    static constexpr uint32_t BUDGET = 227 * 1024 - 4096;
    static constexpr int ring(int vs, int pb)
    {
        return static_cast<int>((BUDGET - (Q_RES + vs * V_STAGE + pb * P_BUF + 1024)) / STAGE);
    }
    // Two P buffers let the softmax write P_(t+1) while P_t V_t still runs;
    // they are used whenever the ring keeps at least three stages (with two V
    // stages for 128-column slices if possible, else one).
    static constexpr int V_DEFAULT = DVS == 128 ? 2 : 1;
    static constexpr bool TWO_P = ring(V_DEFAULT, 2) >= 3 || ring(1, 2) >= 3;
    static constexpr int P_BUFS = TWO_P ? 2 : 1;
    static constexpr int V_STAGES = ring(V_DEFAULT, P_BUFS) >= 3 ? V_DEFAULT : 1;
    static constexpr int STAGES = ring(V_STAGES, P_BUFS);
    static constexpr uint32_t SMEM = Q_RES + V_STAGES * V_STAGE + P_BUFS * P_BUF + 1024 +
                                     STAGES * STAGE;
    static_assert(STAGES >= 3, "too few pipeline stages");
    static_assert(SMEM <= BUDGET, "shared-memory budget exceeded");
};

template <int DVS, bool OUT_F32, int QMODE>
__global__ void __launch_bounds__(kThreads, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, void* O, long long ldo, long long sO,
                     int Nq, int Nk, int dv, int n_chunks, float scale_log2, int o_vec, int zq,
                     int zk, int zv, int dv_slices, int kv_per_split, float* ws_o, float* ws_ml,
                     int hook, unsigned int* err)
{
    using Cfg = AttnCfg<DVS, QMODE>;
    constexpr int VS = Cfg::V_STAGES;
    constexpr int QK_STAGES = Cfg::STAGES;
    constexpr uint32_t QK_STAGE = Cfg::STAGE;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t qk_full[QK_STAGES];
    __shared__ __align__(8) uint64_t qk_empty[QK_STAGES];
    __shared__ __align__(8) uint64_t q_full;              // the resident Q (QMODE > 0)
    __shared__ __align__(8) uint64_t v_full[VS];
    __shared__ __align__(8) uint64_t v_empty[VS];
    __shared__ __align__(8) uint64_t s_full[2];
    __shared__ __align__(8) uint64_t s_empty[2];
    constexpr int PB = Cfg::P_BUFS;
    __shared__ __align__(8) uint64_t p_full[PB];
    __shared__ __align__(8) uint64_t p_empty[PB];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ __align__(8) uint64_t drain_bar2;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float red[2][2][BM];   // per-row partial maxima of the two halves, by block parity
    __shared__ float lsum[2][BM];     // per-row partial normalisers of the two halves

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t q_res = base;                       // resident Q chunks
    const uint32_t qk_base = base + Cfg::Q_RES;        // the ring
    const uint32_t v_base = qk_base + QK_STAGES * QK_STAGE;
    const uint32_t p_base = v_base + VS * Cfg::V_STAGE;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * BM;
    // grid.y walks the output slices and, for a split over the keys, the
    // splits: this CTA takes key blocks kv0 .. kv0 + n_kv - 1
    const int slice = static_cast<int>(blockIdx.y) % dv_slices;
    const int split = static_cast<int>(blockIdx.y) / dv_slices;
    const int dv0 = slice * DVS;
    const int bz = static_cast<int>(blockIdx.z);
    const int kv0 = split * kv_per_split;
    const int n_kv = min((Nk + BN - 1) / BN - kv0, kv_per_split);

    if (threadIdx.x == 0) {
        for (int s = 0; s < QK_STAGES; ++s) {
            mbar_init(smem_u32(&qk_full[s]), 1);
            mbar_init(smem_u32(&qk_empty[s]), 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(smem_u32(&v_full[s]), 1);
            mbar_init(smem_u32(&v_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&s_full[b]), 1);
            mbar_init(smem_u32(&s_empty[b]), kSoftmaxThreads);
        }
        mbar_init(smem_u32(&q_full), 1);
        for (int b = 0; b < PB; ++b) {
            mbar_init(smem_u32(&p_full[b]), kSoftmaxThreads);
            mbar_init(smem_u32(&p_empty[b]), 1);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        mbar_init(smem_u32(&drain_bar2), 1);
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
            bool ok = true;
            if constexpr (QMODE > 0) {
                // the CTA's Q tile, once
                const uint32_t qb = smem_u32(&q_full);
                mbar_arrive_expect_tx(qb, static_cast<uint32_t>(n_chunks) * Q_CHUNK);
                for (int c = 0; c < n_chunks; ++c)
                    tma_load_3d(q_res + c * Q_CHUNK, &tmQ, qb, c * DC, q0, bz * zq);
            }
            for (int t = 0; t < n_kv && ok; ++t) {
                for (int c = 0; c < n_chunks; ++c) {
                    if (!mbar_wait(smem_u32(&qk_empty[s]), ph ^ 1u, &abort_flag)) {
                        abort_flag = 1;
                        atomicOr(err, ERR_ATTENTION);
                        ok = false;
                        break;
                    }
                    if (!(hook == 1 && t == 0 && c == 0)) {  // test hook: leave one stage empty
                        const uint32_t fb = smem_u32(&qk_full[s]);
                        const uint32_t sa = qk_base + s * QK_STAGE;
                        mbar_arrive_expect_tx(fb, QK_STAGE);
                        if constexpr (QMODE == 0) {
                            tma_load_3d(sa, &tmQ, fb, c * DC, q0, bz * zq);
                            tma_load_3d(sa + Q_CHUNK, &tmK, fb, c * DC, (kv0 + t) * BN, bz * zk);
                        } else {
                            tma_load_3d(sa, &tmK, fb, c * DC, (kv0 + t) * BN, bz * zk);
                        }
                        ++issued;
                    }
                    if (++s == QK_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // wait for this thread's copies still in flight before leaving
            for (uint32_t i = 0; i < min(issued, static_cast<uint32_t>(QK_STAGES)); ++i) {
                if (--s < 0) {
                    s = QK_STAGES - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&qk_full[s]), ph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
            if constexpr (QMODE > 0) {
                if (!mbar_wait(smem_u32(&q_full), 0, nullptr)) atomicOr(err, ERR_DRAIN);
            }
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
                const uint32_t sv = v_base + s * Cfg::V_STAGE;
                mbar_arrive_expect_tx(fb, Cfg::V_STAGE);
#pragma unroll
                for (int i = 0; i < DVS / 64; ++i)
                    tma_load_3d(sv + i * V_BOX, &tmV, fb, dv0 + i * 64, (kv0 + t) * BN, bz * zv);
                ++issued;
                if (++s == VS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            for (uint32_t i = 0; i < min(issued, static_cast<uint32_t>(VS)); ++i) {
                if (--s < 0) {
                    s = VS - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&v_full[s]), ph, nullptr)) atomicOr(err, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------ MMA issuer: S = Q K^T
        // (a second issuer, warp 3, does O += P V, so that neither stream
        // of MMAs waits behind the other's barriers)
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(BM, BN, false, false);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            if constexpr (QMODE > 0) {
                ok = mbar_wait(smem_u32(&q_full), 0, &abort_flag);
                tc_fence_after();
            }
            for (int t = 0; t < n_kv && ok; ++t) {
                // S_t into S buffer t % 2, once the softmax has read S_(t-2) from it
                const int sb = t & 1;
                if (!mbar_wait(smem_u32(&s_empty[sb]), ((t >> 1) & 1) ^ 1u, &abort_flag,
                               long_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_s = tmem_base + static_cast<uint32_t>(sb * BN);
                for (int c = 0; c < n_chunks; ++c) {
                    if (!mbar_wait(smem_u32(&qk_full[s]), ph, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = qk_base + s * QK_STAGE;
                    const uint32_t qa = QMODE > 0 ? q_res + c * Q_CHUNK : sa;
                    const uint32_t ka = QMODE > 0 ? sa : sa + Q_CHUNK;
                    // both operands K-major: 8-row groups 1024 B apart, +32 B per 16 of d
                    const uint64_t ad = sdesc_sw128(qa, 16, 1024);
                    const uint64_t bd = sdesc_sw128(ka, 16, 1024);
#pragma unroll
                    for (int k = 0; k < DC / 16; ++k)
                        umma_f16(d_s, ad + 2ull * k, bd + 2ull * k, idesc_s, (c | k) != 0 ? 1u : 0u);
                    umma_commit(smem_u32(&qk_empty[s]));
                    if (++s == QK_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&s_full[sb]));
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
            // every MMA this thread issued must finish before TMEM is freed
            umma_commit(smem_u32(&drain_bar));
            if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------ MMA issuer: O += P V
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_f16_f32(BM, DVS, false, true);
            int vs = 0;
            uint32_t vph = 0;
            bool ok = true;
            for (int u = 0; u < n_kv; ++u) {
                const int pb = u % PB;
                const uint32_t pph = static_cast<uint32_t>((u / PB) & 1);
                if (!mbar_wait(smem_u32(&p_full[pb]), pph, &abort_flag, long_limit) ||
                    !mbar_wait(smem_u32(&v_full[vs]), vph, &abort_flag, long_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P: K-major, two 64-key atoms 16 KB apart.  V: MN-major,
                // 64-column boxes 16 KB apart, 16 keys = 2048 B per step.
                const uint64_t ad = sdesc_sw128(p_base + pb * P_BUF, 16, 1024);
                const uint64_t bd = sdesc_sw128(v_base + vs * Cfg::V_STAGE, V_BOX, 1024);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    umma_f16(tmem_base + O_COL, ad + ((k / 4) * (P_ATOM >> 4) + (k % 4) * 2),
                             bd + 128ull * k, idesc_o, (u | k) != 0 ? 1u : 0u);
                umma_commit(smem_u32(&v_empty[vs]));
                umma_commit(smem_u32(&p_empty[pb]));
                if (++vs == VS) {
                    vs = 0;
                    vph ^= 1u;
                }
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
            umma_commit(smem_u32(&drain_bar2));
            if (!mbar_wait(smem_u32(&drain_bar2), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------- softmax and output
        // Two warps per TMEM lane quadrant: warp h of the pair takes keys
        // h*64 .. h*64+63 of each block and output columns h*DVS/2 ..; the
        // pair agrees on each row's maximum (and, at the end, its sum)
        // through shared memory and a 64-thread named barrier.
        const int q = warp & 3;
        const int h = (warp - 4) >> 2;
        const int r = q * 32 + lane;  // this thread's query row in the tile
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        constexpr int HK = BN / 2;    // keys per warp
        constexpr int HO = DVS / 2;   // output columns per warp
        float m_run = -INFINITY;      // running maximum, base-2 scaled logits
        float l_run = 0.0f;           // this half's share of the running normaliser
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
            const int sb = t & 1;
            uint32_t raw[HK];
            float mine = 0.0f;
            const int valid = min(BN, Nk - (kv0 + t) * BN) - h * HK;
            const bool pos_scale = scale_log2 >= 0.0f;
            if (ok) {
                const bool got =
                    mbar_wait(smem_u32(&s_full[sb]), (t >> 1) & 1, &abort_flag, long_limit);
                if (!__all_sync(0xffffffffu, got)) fail();
            }
            if (ok) {
                tc_fence_after();
                // this half of S_t row r: two 32-column loads in flight, one wait
#pragma unroll
                for (int i = 0; i < HK / 32; ++i)
                    tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(sb * BN + h * HK + 32 * i),
                                       *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * i));
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&s_empty[sb]));
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
            red[sb][h][r] = mine;
            named_bar_sync(1 + q, 64);
            const float other = red[sb][h ^ 1][r];
            if (!ok) continue;

            const float mraw = pos_scale ? fmaxf(mine, other) : fminf(mine, other);
            const float mx = mraw * scale_log2;
            const bool raise = mx > m_run + kRescaleLog2;
            float alpha = 1.0f;
            if (raise) {
                alpha = ex2_approx(m_run - mx);  // 0 for the first block
                l_run *= alpha;
                m_run = mx;
            }
            const float neg_m = -m_run;

            // P = 2^(s * scale * log2 e - m) in fp16 (packed pairs, in
            // registers while the previous block's P V may still run)
            uint32_t pw[HK / 2];
            float l0 = 0.0f, l1 = 0.0f;
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
                    // the normaliser sums the weights the MMA uses: the fp16 ones
                    const float2 r2 = __half22float2(v2);
                    l0 += r2.x;
                    l1 += r2.y;
                    pw[j / 2] = *reinterpret_cast<const uint32_t*>(&v2);
                }
            };
            if (valid < HK) make_p(std::true_type{});
            else make_p(std::false_type{});
            l_run += l0 + l1;

            // P buffer t % PB is free once the MMAs of block t - PB are done
            // (with one buffer that is block t - 1, which also frees O)
            if (t >= PB) {
                const int u = t - PB;
                const bool got_p = mbar_wait(smem_u32(&p_empty[u % PB]), (u / PB) & 1, &abort_flag,
                                             long_limit);
                if (!__all_sync(0xffffffffu, got_p)) {
                    fail();
                    continue;
                }
            }
            if (t > 0 && __any_sync(0xffffffffu, raise)) {
                // O *= alpha (1 in rows that kept their maximum) once the MMAs
                // of block t - 1 are done; with two P buffers that is one more
                // wait, on the buffer of block t - 1
                if (PB == 2) {
                    const int u = t - 1;
                    const bool got_o = mbar_wait(smem_u32(&p_empty[u % PB]), (u / PB) & 1,
                                                 &abort_flag, long_limit);
                    if (!__all_sync(0xffffffffu, got_o)) {
                        fail();
                        continue;
                    }
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < HO; c += 32) {
                    const uint32_t col = O_COL + static_cast<uint32_t>(h * HO + c);
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(t_lane + col, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st_32x32b_x32(t_lane + col, o);
                }
                tmem_st_wait();
            }

            // row r of this half's 64-key atom of the swizzled K-major P tile:
            // 16-byte chunk ch of the row sits at chunk ch ^ (r % 8)
            const uint32_t prow = p_base + static_cast<uint32_t>(t % PB) * P_BUF +
                                  static_cast<uint32_t>(h) * P_ATOM + static_cast<uint32_t>(r) * 128u;
#pragma unroll
            for (int ch = 0; ch < HK / 8; ++ch) {
                const uint32_t pos = static_cast<uint32_t>(ch ^ (r & 7));
                st_shared_v4(prow + pos * 16u, pw[4 * ch], pw[4 * ch + 1], pw[4 * ch + 2],
                             pw[4 * ch + 3]);
            }
            fence_proxy_async_smem();  // generic-proxy P writes -> visible to the tensor core
            tc_fence_before();
            mbar_arrive(smem_u32(&p_full[t % PB]));
        }
        if (ok) {
            // the last block's MMAs complete O
            const int u = n_kv - 1;
            const bool got = mbar_wait(smem_u32(&p_empty[u % PB]), (u / PB) & 1, &abort_flag,
                                       long_limit);
            if (!__all_sync(0xffffffffu, got)) fail();
        }
        // both halves of the row's normaliser (every softmax thread reaches
        // this barrier exactly once)
        lsum[h][r] = l_run;
        named_bar_sync(1 + q, 64);
        const float l_row = lsum[0][r] + lsum[1][r];
        if (ok && ws_o == nullptr) {
            tc_fence_after();
            const float inv_l = 1.0f / l_row;
            const int m = q0 + r;
            void* Ob = batch_ptr(O, bz, sO, OUT_F32 ? 4 : 2);
#pragma unroll 1
            for (int c = 0; c < HO; c += 32) {
                const int cc = h * HO + c;
                uint32_t o[32];
                tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(cc), o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv_l);
                const int n = dv0 + cc;
                if (m < Nq && n < dv) store_chunk<OUT_F32>(Ob, ldo, m, n, dv, o, o_vec != 0);
            }
        } else if (ok) {
            // one split of the keys: the unnormalised O, the running maximum
            // (base 2) and the normaliser go to the workspace for the combine
            tc_fence_after();
            const int m = q0 + r;
            const long long row = (static_cast<long long>(split) * gridDim.z + bz) * Nq + m;
            const int ldw = (dv + 3) & ~3;  // workspace rows padded to 16 bytes
#pragma unroll 1
            for (int c = 0; c < HO; c += 32) {
                const int cc = h * HO + c;
                uint32_t o[32];
                tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(cc), o);
                tmem_ld_wait();
                const int n = dv0 + cc;
                if (m < Nq && n < dv) store_chunk<true>(ws_o + row * ldw, 0, 0, n, dv, o, true);
            }
            if (m < Nq && slice == 0 && h == 0) {
                ws_ml[2 * row] = m_run;
                ws_ml[2 * row + 1] = l_row;
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

// The combine step of a split over the keys: per output element,
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s with M = max_s m_s, the
// same merge of running maxima and normalisers the blockwise pass applies.
// A CTA takes blockDim.y query rows of one batch entry; a thread takes four
// columns at a time.  Two short passes over the splits (the maximum, then
// the weighted sums in split order) keep the registers few, so that many
// rows are in flight per SM.
constexpr int kMaxSplit = 16;

template <bool OUT_F32>
__global__ void __launch_bounds__(256)
attention_combine_kernel(const float* ws_o, const float* ws_ml, void* O, long long ldo,
                         long long sO, int Nq, int dv, int n_split)
{
    const int b = static_cast<int>(blockIdx.z);
    const int batch = static_cast<int>(gridDim.z);
    const int ldw = (dv + 3) & ~3;
    void* Ob = batch_ptr(O, b, sO, OUT_F32 ? 4 : 2);
    for (int m = blockIdx.y * blockDim.y + threadIdx.y; m < Nq; m += gridDim.y * blockDim.y) {
        // the row's largest maximum over the splits
        float M = -INFINITY;
#pragma unroll 4
        for (int sp = 0; sp < n_split; ++sp)
            M = fmaxf(M, ws_ml[2 * ((static_cast<long long>(sp) * batch + b) * Nq + m)]);
        for (int n = 4 * static_cast<int>(threadIdx.x); n < dv; n += 4 * static_cast<int>(blockDim.x)) {
            float den = 0.0f;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int sp = 0; sp < n_split; ++sp) {
                const long long row = (static_cast<long long>(sp) * batch + b) * Nq + m;
                const float w = ex2_approx(ws_ml[2 * row] - M);  // the split's weight
                den = fmaf(w, ws_ml[2 * row + 1], den);
                const float4 ov = *reinterpret_cast<const float4*>(ws_o + row * ldw + n);
                num.x = fmaf(w, ov.x, num.x);
                num.y = fmaf(w, ov.y, num.y);
                num.z = fmaf(w, ov.z, num.z);
                num.w = fmaf(w, ov.w, num.w);
            }
            const float inv = 1.0f / den;
            const float y[4] = {num.x * inv, num.y * inv, num.z * inv, num.w * inv};
            const long long i = static_cast<long long>(m) * ldo + n;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (n + j < dv) {
                    if constexpr (OUT_F32)
                        static_cast<float*>(Ob)[i + j] = y[j];
                    else
                        static_cast<__half*>(Ob)[i + j] = __float2half_rn(y[j]);
                }
            }
        }
    }
}

std::mutex g_attr_mu;
bool g_attr_set[64][12];

template <int DVS, bool OUT_F32, int QMODE>
cudaError_t launch_cfg(const AttnArgs& a)
{
    using Cfg = AttnCfg<DVS, QMODE>;
    auto kernel = attention_fwd_kernel<DVS, OUT_F32, QMODE>;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const int slot = ((DVS == 256 ? 2 : 0) + (OUT_F32 ? 1 : 0)) * 3 + QMODE / 2;
        std::lock_guard<std::mutex> lock(g_attr_mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!g_attr_set[dev][slot]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(Cfg::SMEM));
            if (e != cudaSuccess) return e;
            g_attr_set[dev][slot] = true;
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
    const int dv_slices = (a.dv + DVS - 1) / DVS;
    const int n_kv = (a.Nk + BN - 1) / BN;
    const int n_split = a.n_split > 1 ? a.n_split : 1;
    const int kv_per_split = (n_kv + n_split - 1) / n_split;
    const dim3 grid((a.Nq + BM - 1) / BM, dv_slices * n_split, a.batch);
    if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
    float* ws_o = n_split > 1 ? static_cast<float*>(a.ws) : nullptr;
    float* ws_ml = n_split > 1 ? ws_o + static_cast<long long>(attention_ws_o_floats(a.batch, a.Nq, a.dv, n_split)) : nullptr;
    const float scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)
    const int n_chunks = (a.d + DC - 1) / DC;
    kernel<<<grid, kThreads, Cfg::SMEM, a.stream>>>(tq, tk, tv, a.O, a.ldo, a.sO, a.Nq, a.Nk,
                                                     a.dv, n_chunks, scale_log2, o_vec,
                                                     a.sQ != 0, a.sK != 0, a.sV != 0, dv_slices,
                                                     kv_per_split, ws_o, ws_ml, a.hook, a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n_split == 1) return e;
    // 4 columns per thread across a row (at most 256 threads), the rest of the
    // 256 threads of a CTA on further rows
    int bx = ((a.dv + 3) / 4 + 31) / 32 * 32;
    if (bx > 256) bx = 256;
    const int by = 256 / bx;
    const long long rows = (a.Nq + by - 1) / by;
    const dim3 cgrid(1, static_cast<unsigned>(rows < 65535 ? rows : 65535), a.batch);
    attention_combine_kernel<OUT_F32><<<cgrid, dim3(bx, by), 0, a.stream>>>(
        ws_o, ws_ml, a.O, a.ldo, a.sO, a.Nq, a.dv, n_split);
    return cudaGetLastError();
}

template <int DVS, bool OUT_F32>
cudaError_t launch_q(const AttnArgs& a)
{
    if (a.d <= 128) return launch_cfg<DVS, OUT_F32, 2>(a);
    if (a.d <= 256) return launch_cfg<DVS, OUT_F32, 4>(a);
    return launch_cfg<DVS, OUT_F32, 0>(a);
}

}  // namespace

namespace {

// Scratch for tg_attention_noalloc: file-scope device memory, so that entry
// point allocates nothing.  16 MB holds the key-split partials of the
// largest calls that split (for example the page's one 1024 x 768 head needs
// 12.6 MB); larger needs are rejected.  Every call on a device uses the same
// bytes.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64];

}  // namespace

void* attention_static_scratch(size_t* bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        // the symbol's address on this device, looked up once
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    *bytes = kStaticScratchBytes;
    return g_scratch_addr[dev];
}

long long attention_ws_o_floats(int batch, int Nq, int dv, int n_split)
{
    // the O partials (rows padded to 4 floats), rounded up to 64 floats so
    // the maxima/normalisers that follow start 256-byte aligned
    const long long n = static_cast<long long>(n_split) * batch * Nq * ((dv + 3) & ~3);
    return (n + 63) / 64 * 64;
}

int attention_splits(int batch, int Nq, int Nk, int dv, int num_sms)
{
    const long long base = static_cast<long long>((Nq + BM - 1) / BM) *
                           ((dv + (dv <= 128 ? 128 : 256) - 1) / (dv <= 128 ? 128 : 256)) * batch;
    const int n_kv = (Nk + BN - 1) / BN;
    if (2 * base > num_sms || n_kv < 2) return 1;
    // as many splits as keep every CTA of the call in one wave (at most 16)
    int want = static_cast<int>(num_sms / base);
    if (want > n_kv) want = n_kv;
    if (want > kMaxSplit) want = kMaxSplit;
    const int per = (n_kv + want - 1) / want;
    return (n_kv + per - 1) / per;
}

size_t attention_ws_bytes(int batch, int Nq, int Nk, int dv, int num_sms)
{
    const int n_split = attention_splits(batch, Nq, Nk, dv, num_sms);
    if (n_split <= 1) return 0;
    return (static_cast<size_t>(attention_ws_o_floats(batch, Nq, dv, n_split)) +
            2ull * n_split * batch * Nq) * sizeof(float);
}

int attention_kernel_choice(int batch, int Nq, int Nk, int d, int dv, int num_sms, bool split_ok,
                            int forced)
{
    const bool tmem_ok = attention_tmem_p_serves(d, dv);
    if (forced == 3 && tmem_ok) return 3;
    if (split_ok && attention_splits(batch, Nq, Nk, dv, num_sms) > 1) return 2;
    return forced == 1 || !tmem_ok ? 1 : 3;
}

cudaError_t launch_attention(const AttnArgs& a)
{
    if (a.tmem_p) return launch_attention_tmem_p(a);
    if (a.dv <= 128) return a.out_f32 ? launch_q<128, true>(a) : launch_q<128, false>(a);
    return a.out_f32 ? launch_q<256, true>(a) : launch_q<256, false>(a);
}

}  // namespace tg

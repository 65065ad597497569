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
// The MMA issuer computes S_(t+1) before P_t V_t, so the tensor core works
// on the next scores while the softmax warps turn S_t into P_t.  The running
// maximum is raised only when a block's maximum exceeds it by more than 8 (in
// base 2): then O (in TMEM) and L are scaled by 2^(m_old - m_new); otherwise
// the stale maximum stays, the probabilities stay below 2^8, and the final
// O / L is the same quotient.  Outputs wider than 256 columns take several
// CTAs, each recomputing S for its own slice of V.
//
// Warp roles (256 threads): 0 TMA for Q and K, 1 TMEM allocation and MMA
// issue, 2 TMA for V, 4-7 softmax and output (warp w reads TMEM lane
// quadrant w % 4).  Every wait is bounded: on expiry a role records it in
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
constexpr int QK_STAGES = 3;
constexpr uint32_t Q_CHUNK = BM * DC * 2;     // 16 KB
constexpr uint32_t K_CHUNK = BN * DC * 2;     // 16 KB
constexpr uint32_t QK_STAGE = Q_CHUNK + K_CHUNK;
constexpr uint32_t P_ATOM = BM * 128;         // [128 rows][64 keys] fp16, 16 KB
constexpr uint32_t P_BUF = 2 * P_ATOM;        // 128 keys
constexpr uint32_t V_BOX = BN * 128;          // [128 keys][64 columns] fp16, 16 KB
constexpr uint32_t TMEM_COLS = 512;           // S0, S1 (128 each), O (<= 256)
constexpr uint32_t O_COL = 256;
constexpr int kThreads = 256;
constexpr uint32_t kSoftmaxThreads = 128;
constexpr float kRescaleLog2 = 8.0f;          // raise the running max past 2^8 growth

template <int DVS>
struct AttnCfg {
    static_assert(DVS == 128 || DVS == 256, "an output slice is 128 or 256 columns");
    static constexpr int V_STAGES = DVS == 128 ? 2 : 1;
    static constexpr uint32_t V_STAGE = BN * DVS * 2;
    static constexpr uint32_t SMEM =
        QK_STAGES * QK_STAGE + V_STAGES * V_STAGE + 2 * P_BUF + 1024;
    static_assert(SMEM <= 227 * 1024, "shared-memory budget exceeded");
};

template <int DVS, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, void* O, long long ldo, long long sO,
                     int Nq, int Nk, int dv, int n_chunks, float scale_log2, int o_vec, int zq,
                     int zk, int zv, int hook, unsigned int* err)
{
    using Cfg = AttnCfg<DVS>;
    constexpr int VS = Cfg::V_STAGES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t qk_full[QK_STAGES];
    __shared__ __align__(8) uint64_t qk_empty[QK_STAGES];
    __shared__ __align__(8) uint64_t v_full[VS];
    __shared__ __align__(8) uint64_t v_empty[VS];
    __shared__ __align__(8) uint64_t s_full[2];
    __shared__ __align__(8) uint64_t s_empty[2];
    __shared__ __align__(8) uint64_t p_full[2];
    __shared__ __align__(8) uint64_t p_empty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t qk_base = base;
    const uint32_t v_base = base + QK_STAGES * QK_STAGE;
    const uint32_t p_base = v_base + VS * Cfg::V_STAGE;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * BM;
    const int dv0 = blockIdx.y * DVS;
    const int bz = static_cast<int>(blockIdx.z);
    const int n_kv = (Nk + BN - 1) / BN;

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
            mbar_init(smem_u32(&p_full[b]), kSoftmaxThreads);
            mbar_init(smem_u32(&p_empty[b]), 1);
        }
        mbar_init(smem_u32(&drain_bar), 1);
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
                        tma_load_3d(sa, &tmQ, fb, c * DC, q0, bz * zq);
                        tma_load_3d(sa + Q_CHUNK, &tmK, fb, c * DC, t * BN, bz * zk);
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
                    tma_load_3d(sv + i * V_BOX, &tmV, fb, dv0 + i * 64, t * BN, bz * zv);
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
        // --------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_f16_f32(BM, DVS, false, true);
            int s = 0, vs = 0;
            uint32_t ph = 0, vph = 0;
            bool ok = true;
            for (int t = 0; t <= n_kv && ok; ++t) {
                if (t < n_kv) {
                    // S_t = Q K_t^T into S buffer t % 2, once the softmax has
                    // read S_(t-2) from it
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
                        // both operands K-major: 8-row groups 1024 B apart, +32 B per 16 of d
                        const uint64_t ad = sdesc_sw128(sa, 16, 1024);
                        const uint64_t bd = sdesc_sw128(sa + Q_CHUNK, 16, 1024);
#pragma unroll
                        for (int k = 0; k < DC / 16; ++k)
                            umma_f16(d_s, ad + 2ull * k, bd + 2ull * k, idesc_s,
                                     (c | k) != 0 ? 1u : 0u);
                        umma_commit(smem_u32(&qk_empty[s]));
                        if (++s == QK_STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&s_full[sb]));
                }
                if (t >= 1) {
                    // O += P_u V_u for the previous block u
                    const int u = t - 1;
                    const int pb = u & 1;
                    if (!mbar_wait(smem_u32(&p_full[pb]), (u >> 1) & 1, &abort_flag, long_limit) ||
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
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(err, ERR_ATTENTION);
            }
            // every MMA issued must finish before TMEM is freed
            umma_commit(smem_u32(&drain_bar));
            if (!mbar_wait(smem_u32(&drain_bar), 0, nullptr)) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------- softmax and output
        const int q = warp & 3;
        const int r = q * 32 + lane;  // this thread's query row in the tile
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        float m_run = -INFINITY;      // running maximum, base-2 scaled logits
        float l_run = 0.0f;           // running normaliser
        bool ok = true;
        for (int t = 0; t < n_kv && ok; ++t) {
            const int sb = t & 1;
            const bool got = mbar_wait(smem_u32(&s_full[sb]), (t >> 1) & 1, &abort_flag, long_limit);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // S_t row r: four 32-column loads in flight, one wait
            uint32_t raw[BN];
#pragma unroll
            for (int i = 0; i < BN / 32; ++i)
                tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(sb * BN + 32 * i),
                                   *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * i));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&s_empty[sb]));

            // block maximum of the base-2 logits; keys past Nk (zero-filled by
            // TMA) are masked, which only the last block can need
            const int valid = min(BN, Nk - t * BN);
            if (valid < BN) {
#pragma unroll
                for (int j = 0; j < BN; ++j)
                    if (j >= valid) raw[j] = __float_as_uint(scale_log2 >= 0.0f ? -INFINITY : INFINITY);
            }
            // (four independent chains keep the reduction short)
            float mc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) mc[c] = __uint_as_float(raw[c]);
            if (scale_log2 >= 0.0f) {
#pragma unroll
                for (int j = 4; j < BN; ++j) mc[j & 3] = fmaxf(mc[j & 3], __uint_as_float(raw[j]));
            } else {
#pragma unroll
                for (int j = 4; j < BN; ++j) mc[j & 3] = fminf(mc[j & 3], __uint_as_float(raw[j]));
            }
            const float mraw = scale_log2 >= 0.0f ? fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]))
                                                  : fminf(fminf(mc[0], mc[1]), fminf(mc[2], mc[3]));
            const float mx = mraw * scale_log2;
            const bool raise = mx > m_run + kRescaleLog2;
            float alpha = 1.0f;
            if (raise) {
                alpha = ex2_approx(m_run - mx);  // 0 for the first block
                l_run *= alpha;
                m_run = mx;
            }
            const float neg_m = -m_run;

            // the P buffer must be free: the MMAs of block t - 2 have read it
            const bool got_p = mbar_wait(smem_u32(&p_empty[sb]), ((t >> 1) & 1) ^ 1u, &abort_flag,
                                         long_limit);
            if (!__all_sync(0xffffffffu, got_p)) {
                ok = false;
                break;
            }
            if (t > 0 && __any_sync(0xffffffffu, raise)) {
                // O *= alpha, after the MMAs of block t - 1 have finished
                const int u = t - 1;
                const bool got_o = mbar_wait(smem_u32(&p_empty[u & 1]), (u >> 1) & 1, &abort_flag,
                                             long_limit);
                if (!__all_sync(0xffffffffu, got_o)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < DVS; c += 32) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(c), o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(c), o);
                }
                tmem_st_wait();
            }

            // P = 2^(s * scale * log2 e - m) in fp16, row r of the swizzled
            // K-major tile; the row sum in two chains.  Masked keys (the last
            // block only) get probability 0 whatever the scale.
            const uint32_t prow = p_base + sb * P_BUF + static_cast<uint32_t>(r) * 128u;
            float l0 = 0.0f, l1 = 0.0f;
            auto write_p = [&](auto masked) {
#pragma unroll
                for (int ch = 0; ch < BN / 8; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int j = 8 * ch + 2 * h;
                        float a0 = fmaf(__uint_as_float(raw[j]), scale_log2, neg_m);
                        float a1 = fmaf(__uint_as_float(raw[j + 1]), scale_log2, neg_m);
                        if constexpr (decltype(masked)::value) {
                            if (j >= valid) a0 = -INFINITY;
                            if (j + 1 >= valid) a1 = -INFINITY;
                        }
                        const float p0 = ex2_approx(a0);
                        const float p1 = ex2_approx(a1);
                        l0 += p0;
                        l1 += p1;
                        __half2 v2 = __floats2half2_rn(p0, p1);
                        w[h] = *reinterpret_cast<uint32_t*>(&v2);
                    }
                    const uint32_t atom = static_cast<uint32_t>(ch >> 3);
                    const uint32_t pos = static_cast<uint32_t>((ch & 7) ^ (r & 7));
                    st_shared_v4(prow + atom * P_ATOM + pos * 16u, w[0], w[1], w[2], w[3]);
                }
            };
            if (valid < BN) write_p(std::true_type{});
            else write_p(std::false_type{});
            l_run += l0 + l1;
            fence_proxy_async_smem();  // generic-proxy P writes -> visible to the tensor core
            tc_fence_before();
            mbar_arrive(smem_u32(&p_full[sb]));
        }
        if (ok) {
            // the last block's MMAs complete O; normalise and store
            const int u = n_kv - 1;
            const bool got = mbar_wait(smem_u32(&p_empty[u & 1]), (u >> 1) & 1, &abort_flag,
                                       long_limit);
            ok = __all_sync(0xffffffffu, got);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.0f / l_run;
            const int m = q0 + r;
            void* Ob = batch_ptr(O, bz, sO, OUT_F32 ? 4 : 2);
#pragma unroll 1
            for (int c = 0; c < DVS; c += 32) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(t_lane + O_COL + static_cast<uint32_t>(c), o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv_l);
                const int n = dv0 + c;
                if (m < Nq && n < dv) store_chunk<OUT_F32>(Ob, ldo, m, n, dv, o, o_vec != 0);
            }
        } else if (lane == 0) {
            abort_flag = 1;
            atomicOr(err, ERR_ATTENTION);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

std::mutex g_attr_mu;
bool g_attr_set[64][4];

template <int DVS, bool OUT_F32>
cudaError_t launch_cfg(const AttnArgs& a)
{
    using Cfg = AttnCfg<DVS>;
    auto kernel = attention_fwd_kernel<DVS, OUT_F32>;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const int slot = (DVS == 256 ? 2 : 0) + (OUT_F32 ? 1 : 0);
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
    const dim3 grid((a.Nq + BM - 1) / BM, (a.dv + DVS - 1) / DVS, a.batch);
    if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
    const float scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)
    const int n_chunks = (a.d + DC - 1) / DC;
    kernel<<<grid, kThreads, Cfg::SMEM, a.stream>>>(tq, tk, tv, a.O, a.ldo, a.sO, a.Nq, a.Nk,
                                                     a.dv, n_chunks, scale_log2, o_vec,
                                                     a.sQ != 0, a.sK != 0, a.sV != 0, a.hook,
                                                     a.err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a)
{
    if (a.dv <= 128) return a.out_f32 ? launch_cfg<128, true>(a) : launch_cfg<128, false>(a);
    return a.out_f32 ? launch_cfg<256, true>(a) : launch_cfg<256, false>(a);
}

}  // namespace tg

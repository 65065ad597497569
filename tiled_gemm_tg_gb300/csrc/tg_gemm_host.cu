// tg_gemm_host.cu -- the C ABI: argument validation, path selection, tensor-
// map encoding and the device error word.  Every check here runs on the host
// before any CUDA call, so invalid arguments never reach the GPU.
//
// The operation is C = A x B (row-major), the running example of the
// TileLang pages ("企业官网建设流程全解析" (cf-1.com) §3.3; "TileLang实战"
// (gsyq.cn) §3.1 and §3.3).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tg_gemm.h"
#include "tg_internal.h"

// One error word per device: kernels OR a bit into it when they abandon a
// bounded wait; tg_gemm_check reads and clears it.
static __device__ unsigned int g_tg_error_word;

namespace {

constexpr int kMaxDevices = 64;
// Largest M, N or K: tile origins (up to a dimension plus one tile) and TMA
// coordinates stay within int32.
constexpr int64_t kMaxDim = 2147483647LL - 1023;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    unsigned int* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int> g_force_path{0};
std::atomic<int> g_test_hook{0};
std::atomic<int> g_force_bn{0};
std::atomic<int> g_force_group{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

tg_status device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tg_error_word) != cudaSuccess) return TG_ERR_CUDA;
        s.err = static_cast<unsigned int*>(p);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return TG_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        s.ready = true;
    }
    *out = &s;
    return TG_OK;
}

size_t esize(tg_dtype t) { return t == TG_F16 ? 2 : 4; }

using u128 = unsigned __int128;

// Byte span [lo, hi) touched by a rows x cols row-major matrix with stride ld
// (rows, cols >= 1).  Computed in 128 bits so no product can wrap.
void span(const void* p, int64_t rows, int64_t cols, int64_t ld, size_t es, u128* lo, u128* hi)
{
    *lo = static_cast<u128>(reinterpret_cast<uintptr_t>(p));
    *hi = *lo + (static_cast<u128>(rows - 1) * static_cast<u128>(ld) + static_cast<u128>(cols)) *
                    static_cast<u128>(es);
}

bool overlaps(u128 a0, u128 a1, u128 b0, u128 b1) { return a0 < b1 && b0 < a1; }

// Validation shared by tg_gemm and tg_gemm_path.  On TG_OK, *path is the
// path the arguments call for (ignoring any forced path).
tg_status classify(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                   int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype,
                   int* path)
{
    *path = tg::PATH_NONE;
    if (M < 0 || N < 0 || K < 0) return TG_ERR_INVALID_ARG;
    const bool pair_ok = (in_dtype == TG_F16 && (out_dtype == TG_F16 || out_dtype == TG_F32)) ||
                         (in_dtype == TG_F32 && out_dtype == TG_F32);
    if (!pair_ok) return TG_ERR_UNSUPPORTED;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TG_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr || ldc < N) return TG_ERR_INVALID_ARG;
    // Every element access is naturally aligned: a pointer that is not a
    // multiple of its element size is rejected rather than handed to a kernel.
    if (reinterpret_cast<uintptr_t>(C) % esize(out_dtype) != 0) return TG_ERR_INVALID_ARG;
    if (K == 0) {
        *path = tg::PATH_ZERO;
        return TG_OK;
    }
    if (A == nullptr || B == nullptr || lda < K || ldb < N) return TG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(A) % esize(in_dtype) != 0 ||
        reinterpret_cast<uintptr_t>(B) % esize(in_dtype) != 0)
        return TG_ERR_INVALID_ARG;
    u128 c0, c1, a0, a1, b0, b1;
    span(C, M, N, ldc, esize(out_dtype), &c0, &c1);
    span(A, M, K, lda, esize(in_dtype), &a0, &a1);
    span(B, K, N, ldb, esize(in_dtype), &b0, &b1);
    const u128 top = static_cast<u128>(1) << 64;  // a span past the address space cannot exist
    if (c1 > top || a1 > top || b1 > top) return TG_ERR_INVALID_ARG;
    if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TG_ERR_INVALID_ARG;

    if (in_dtype == TG_F32) {
        *path = tg::PATH_SIMT;
        return TG_OK;
    }
    // The TMA engine needs 16-byte aligned bases and row strides that are
    // multiples of 16 bytes (and below 2^40 bytes).
    const int64_t kMaxTmaLd = int64_t(1) << 38;
    const bool tma_ok = (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (lda % 8 == 0) &&
                        (ldb % 8 == 0) && lda < kMaxTmaLd && ldb < kMaxTmaLd;
    if (!tma_ok) {
        *path = tg::PATH_BOUNDARY;
    } else if (M <= tg::kSkinnyMaxM) {
        *path = tg::PATH_SKINNY;
    } else if (tg::pair_tiles(static_cast<int>(M), static_cast<int>(N)) >= tg::kPairMinTiles) {
        *path = tg::PATH_MAIN_PAIR;
    } else {
        *path = tg::PATH_MAIN;
    }
    return TG_OK;
}

bool path_serves(int path, int natural, tg_dtype in_dtype, int64_t M)
{
    if (path == natural) return true;
    if (natural == tg::PATH_ZERO || natural == tg::PATH_NONE) return false;
    switch (path) {
        case tg::PATH_SIMT: return in_dtype == TG_F32;
        case tg::PATH_BOUNDARY: return in_dtype == TG_F16;
        case tg::PATH_MAIN:
        case tg::PATH_MAIN_PAIR:
            return in_dtype == TG_F16 && natural != tg::PATH_BOUNDARY;
        case tg::PATH_SKINNY:
            return in_dtype == TG_F16 && natural != tg::PATH_BOUNDARY && M <= tg::kSkinnyMaxM;
        default: return false;
    }
}

// Validates the fused-epilogue arguments of tg_gemm_ex against C (M, N >= 1,
// C already validated) and fills *e.  D may be C itself (same base and row
// stride: an in-place update); any other overlap of D or bias with C is an
// error, as is a pointer that is not a multiple of its element size.
tg_status classify_epilogue(int64_t M, int64_t N, void* C, int64_t ldc, tg_dtype out_dtype,
                            float alpha, float beta, const void* D, int64_t ldd,
                            const float* bias, int act, tg::Epilogue* e)
{
    if (act != tg::ACT_NONE && act != tg::ACT_RELU && act != tg::ACT_GELU) return TG_ERR_INVALID_ARG;
    const size_t es = esize(out_dtype);
    u128 c0, c1;
    span(C, M, N, ldc, es, &c0, &c1);
    const u128 top = static_cast<u128>(1) << 64;
    if (beta != 0.0f) {
        if (D == nullptr || ldd < N || reinterpret_cast<uintptr_t>(D) % es != 0)
            return TG_ERR_INVALID_ARG;
        u128 d0, d1;
        span(D, M, N, ldd, es, &d0, &d1);
        if (d1 > top) return TG_ERR_INVALID_ARG;
        const bool in_place = (D == C && ldd == ldc);
        if (!in_place && overlaps(c0, c1, d0, d1)) return TG_ERR_INVALID_ARG;
    }
    if (bias != nullptr) {
        if (reinterpret_cast<uintptr_t>(bias) % 4 != 0) return TG_ERR_INVALID_ARG;
        u128 b0, b1;
        span(bias, 1, N, N, 4, &b0, &b1);
        if (b1 > top || overlaps(c0, c1, b0, b1)) return TG_ERR_INVALID_ARG;
    }
    e->alpha = alpha;
    e->beta = beta;
    e->D = beta != 0.0f ? D : nullptr;
    e->ldd = beta != 0.0f ? ldd : 0;
    e->bias = bias;
    e->act = act;
    e->on = !(alpha == 1.0f && beta == 0.0f && bias == nullptr && act == tg::ACT_NONE);
    e->d_vec = beta != 0.0f && reinterpret_cast<uintptr_t>(D) % 16 == 0 &&
               (static_cast<size_t>(ldd) * es) % 16 == 0;
    e->bias_vec = bias != nullptr && reinterpret_cast<uintptr_t>(bias) % 16 == 0;
    return TG_OK;
}

// The body of tg_gemm and tg_gemm_ex once the arguments have been classified.
tg_status run(int path, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
              const void* B, int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype,
              tg_dtype out_dtype, const tg::Epilogue& epi, tg_stream_t stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == tg::PATH_ZERO && !epi.on) {
        const size_t es = esize(out_dtype);
        cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * es, 0,
                                          static_cast<size_t>(N) * es, static_cast<size_t>(M), s);
        return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    if (path != tg::PATH_ZERO) {
        const int forced = g_force_path.load(std::memory_order_relaxed);
        if (forced != 0) {
            if (!path_serves(forced, path, in_dtype, M)) return TG_ERR_UNSUPPORTED;
            path = forced;
        }
    }

    DeviceState* ds = nullptr;
    tg_status st = device_state(&ds);
    if (st != TG_OK) return st;

    tg::GemmArgs a;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.A = A;
    a.lda = lda;
    a.B = B;
    a.ldb = ldb;
    a.C = C;
    a.ldc = ldc;
    a.out_f32 = (out_dtype == TG_F32);
    a.err = ds->err;
    a.hook = g_test_hook.load(std::memory_order_relaxed);
    a.group_m = g_force_group.load(std::memory_order_relaxed);
    a.num_sms = ds->num_sms;
    a.stream = s;
    a.epi = epi;

    cudaError_t e = cudaSuccess;
    switch (path) {
        case tg::PATH_ZERO: e = tg::launch_epilogue_only(a); break;
        case tg::PATH_SIMT: e = tg::launch_simt_f32(a); break;
        case tg::PATH_MAIN: {
            const int bn = g_force_bn.load(std::memory_order_relaxed);
            e = tg::launch_main(a, bn != 0 ? bn : tg::main_tile_n(a.M, a.N, a.num_sms));
            break;
        }
        case tg::PATH_BOUNDARY: e = tg::launch_boundary(a); break;
        case tg::PATH_MAIN_PAIR: e = tg::launch_main_pair(a); break;
        case tg::PATH_SKINNY: e = tg::launch_skinny(a); break;
        default: return TG_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace

namespace tg {

bool encode_tmap_f16(CUtensorMap* map, const void* ptr, uint64_t cols, uint64_t rows, uint64_t ld,
                     uint32_t box_cols, uint32_t box_rows)
{
    if (!g_encode) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tg

extern "C" {

tg_status tg_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                  int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype,
                  tg_stream_t stream)
{
    int path = tg::PATH_NONE;
    tg_status st = classify(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, &path);
    if (st != TG_OK || path == tg::PATH_NONE) return st;
    return run(path, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, tg::Epilogue{}, stream);
}

tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype,
                     float alpha, float beta, const void* D, int64_t ldd, const float* bias,
                     tg_activation act, tg_stream_t stream)
{
    if (act != TG_ACT_NONE && act != TG_ACT_RELU && act != TG_ACT_GELU) return TG_ERR_INVALID_ARG;
    int path = tg::PATH_NONE;
    tg_status st = classify(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, &path);
    if (st != TG_OK || path == tg::PATH_NONE) return st;
    tg::Epilogue epi;
    st = classify_epilogue(M, N, C, ldc, out_dtype, alpha, beta, D, ldd, bias,
                           static_cast<int>(act), &epi);
    if (st != TG_OK) return st;
    return run(path, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epi, stream);
}

tg_status tg_gemm_check(tg_stream_t stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return TG_ERR_CUDA;
    DeviceState* ds = nullptr;
    tg_status st = device_state(&ds);
    if (st != TG_OK) return st;
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, ds->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return TG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TG_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(ds->err, 0, sizeof(word), s) != cudaSuccess) return TG_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return TG_ERR_CUDA;
        return TG_ERR_TIMEOUT;
    }
    return TG_OK;
}

const char* tg_status_string(tg_status status)
{
    switch (status) {
        case TG_OK: return "TG_OK";
        case TG_ERR_INVALID_ARG: return "TG_ERR_INVALID_ARG";
        case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
        case TG_ERR_CUDA: return "TG_ERR_CUDA";
        case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
    }
    return "TG_ERR_UNKNOWN";
}

int tg_gemm_path(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype)
{
    int path = tg::PATH_NONE;
    if (classify(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, &path) != TG_OK)
        return tg::PATH_NONE;
    const int forced = g_force_path.load(std::memory_order_relaxed);
    if (forced != 0 && path != tg::PATH_ZERO && path != tg::PATH_NONE)
        return path_serves(forced, path, in_dtype, M) ? forced : tg::PATH_NONE;
    return path;
}

void tg_gemm_force_path(int path)
{
    if (path < 0 || path > tg::PATH_MAIN_PAIR || path == tg::PATH_ZERO) path = 0;
    g_force_path.store(path, std::memory_order_relaxed);
}

void tg_gemm_test_hook(int hook) { g_test_hook.store(hook == 1 ? 1 : 0, std::memory_order_relaxed); }

tg_status tg_gemm_force_tiling(int bn, int group_m)
{
    if (!(bn == 0 || bn == 64 || bn == 128 || bn == 256)) return TG_ERR_INVALID_ARG;
    if (group_m < 0 || group_m > 64) return TG_ERR_INVALID_ARG;
    g_force_bn.store(bn, std::memory_order_relaxed);
    g_force_group.store(group_m, std::memory_order_relaxed);
    return TG_OK;
}

int tg_gemm_version(void) { return 100; }

}  // extern "C"

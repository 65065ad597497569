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
// Largest batch: the kernels that walk a batch over grid.z allow 65535.
constexpr int64_t kMaxBatch = 65535;

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
std::atomic<int> g_force_split_k{0};
std::atomic<int> g_force_group{0};
std::atomic<int> g_force_attn{0};
std::atomic<int> g_force_split_tail{-1};
std::atomic<int> g_force_stages{0};
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

size_t esize(tg_dtype t) { return t == TG_F16 ? 2 : t == TG_E4M3 ? 1 : 4; }

using u128 = unsigned __int128;

// Byte span [lo, hi) touched by `batch` rows x cols row-major matrices with
// row stride ld and matrix stride `stride` (rows, cols, batch >= 1).
// Computed in 128 bits so no product can wrap.
void span(const void* p, int64_t rows, int64_t cols, int64_t ld, size_t es, u128* lo, u128* hi,
          int64_t batch = 1, int64_t stride = 0)
{
    *lo = static_cast<u128>(reinterpret_cast<uintptr_t>(p));
    *hi = *lo + (static_cast<u128>(batch - 1) * static_cast<u128>(stride) +
                 static_cast<u128>(rows - 1) * static_cast<u128>(ld) + static_cast<u128>(cols)) *
                    static_cast<u128>(es);
}

bool overlaps(u128 a0, u128 a1, u128 b0, u128 b1) { return a0 < b1 && b0 < a1; }

// One call's arguments: `batch` products C_b = A_b x B_b, X_b = X + b * sX
// elements (batch 1 and strides 0 for tg_gemm).
struct Problem {
    int64_t batch, M, N, K;
    const void* A;
    int64_t lda, sA;
    const void* B;
    int64_t ldb, sB;
    void* C;
    int64_t ldc, sC;
    tg_dtype in_dtype, out_dtype;
};

// The TMA engine addresses a batch of matrices through a 3-D tensor map:
// a matrix stride that is a multiple of 16 bytes, below 2^40 bytes and at
// least one whole matrix (or 0, one matrix broadcast to every b).
bool tma_stride_ok(int64_t stride, int64_t rows, int64_t ld, int64_t es)
{
    if (stride == 0) return true;
    return stride < (int64_t(1) << 39) / es && (stride * es) % 16 == 0 &&
           static_cast<u128>(stride) >= static_cast<u128>(rows) * static_cast<u128>(ld);
}

// Whether a problem with `tiles` 256 x 256 tiles and depth K goes to the
// pair kernel (M, N and K already past their minimums).
bool pair_worth(int64_t tiles, int64_t K)
{
    return tiles >= tg::kPairMinTilesShortK || (tiles >= tg::kPairMinTiles && K >= tg::kPairLongK);
}

// Validation shared by every entry point.  On TG_OK, *path is the path the
// arguments call for (ignoring any forced path).
tg_status classify(const Problem& p, int* path)
{
    *path = tg::PATH_NONE;
    const int64_t M = p.M, N = p.N, K = p.K;
    if (M < 0 || N < 0 || K < 0 || p.batch < 0) return TG_ERR_INVALID_ARG;
    if (p.sA < 0 || p.sB < 0 || p.sC < 0) return TG_ERR_INVALID_ARG;
    const bool pair_ok =
        ((p.in_dtype == TG_F16 || p.in_dtype == TG_E4M3) &&
         (p.out_dtype == TG_F16 || p.out_dtype == TG_F32)) ||
        (p.in_dtype == TG_F32 && p.out_dtype == TG_F32);
    if (!pair_ok) return TG_ERR_UNSUPPORTED;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || p.batch > kMaxBatch)
        return TG_ERR_UNSUPPORTED;
    if (M == 0 || N == 0 || p.batch == 0) return TG_OK;
    // every tile index of the whole batch fits in 32 bits
    if (((M + 127) / 128) * ((N + 63) / 64) * p.batch >= (int64_t(1) << 31))
        return TG_ERR_UNSUPPORTED;
    if (p.C == nullptr || p.ldc < N) return TG_ERR_INVALID_ARG;
    // the matrices of C are disjoint
    if (p.batch > 1 && p.sC < (M - 1) * p.ldc + N) return TG_ERR_INVALID_ARG;
    // Every element access is naturally aligned: a pointer that is not a
    // multiple of its element size is rejected rather than handed to a kernel.
    const size_t ei = esize(p.in_dtype), eo = esize(p.out_dtype);
    if (reinterpret_cast<uintptr_t>(p.C) % eo != 0) return TG_ERR_INVALID_ARG;
    u128 c0, c1;
    span(p.C, M, N, p.ldc, eo, &c0, &c1, p.batch, p.sC);
    const u128 top = static_cast<u128>(1) << 64;  // a span past the address space cannot exist
    if (c1 > top) return TG_ERR_INVALID_ARG;
    if (K == 0) {
        *path = tg::PATH_ZERO;
        return TG_OK;
    }
    if (p.A == nullptr || p.B == nullptr || p.lda < K || p.ldb < N) return TG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p.A) % ei != 0 || reinterpret_cast<uintptr_t>(p.B) % ei != 0)
        return TG_ERR_INVALID_ARG;
    u128 a0, a1, b0, b1;
    span(p.A, M, K, p.lda, ei, &a0, &a1, p.batch, p.sA);
    span(p.B, K, N, p.ldb, ei, &b0, &b1, p.batch, p.sB);
    if (a1 > top || b1 > top) return TG_ERR_INVALID_ARG;
    if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TG_ERR_INVALID_ARG;

    if (p.in_dtype == TG_F32) {
        *path = tg::PATH_SIMT;
        return TG_OK;
    }
    // The TMA engine needs 16-byte aligned bases and row strides that are
    // multiples of 16 bytes (and below 2^40 bytes).
    const int64_t e = static_cast<int64_t>(ei);
    const int64_t kMaxTmaLdBytes = int64_t(1) << 39;
    // (sizes are compared before they are multiplied, so nothing can overflow)
    const bool tma_ok = (reinterpret_cast<uintptr_t>(p.A) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(p.B) % 16 == 0) &&
                        p.lda < kMaxTmaLdBytes / e && p.ldb < kMaxTmaLdBytes / e &&
                        (p.lda * e) % 16 == 0 && (p.ldb * e) % 16 == 0 &&
                        (p.batch == 1 || (tma_stride_ok(p.sA, M, p.lda, e) &&
                                          tma_stride_ok(p.sB, K, p.ldb, e)));
    const bool e4m3 = p.in_dtype == TG_E4M3;
    // E4M3 runs on the TMA kernels only (the skinny and boundary kernels are
    // fp16): operands the TMA engine cannot address are not supported.
    if (e4m3 && !tma_ok) return TG_ERR_UNSUPPORTED;
    if (!tma_ok) {
        *path = tg::PATH_BOUNDARY;
    } else if (M <= tg::kSkinnyMaxM && !e4m3) {
        *path = tg::PATH_SKINNY;
    } else if (M >= tg::kPairMinMN && N >= tg::kPairMinMN && K >= tg::kPairMinK &&
               pair_worth(static_cast<int64_t>(tg::pair_tiles(static_cast<int>(M),
                                                              static_cast<int>(N))) * p.batch,
                          K)) {
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
    if (in_dtype == TG_E4M3) return path == tg::PATH_MAIN || path == tg::PATH_MAIN_PAIR;
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

// The body of every entry point once the arguments have been classified.
tg_status run(int path, const Problem& p, const tg::Epilogue& epi, tg_stream_t stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == tg::PATH_ZERO && !epi.on && p.batch == 1) {
        const size_t es = esize(p.out_dtype);
        cudaError_t e = cudaMemset2DAsync(p.C, static_cast<size_t>(p.ldc) * es, 0,
                                          static_cast<size_t>(p.N) * es,
                                          static_cast<size_t>(p.M), s);
        return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    if (path != tg::PATH_ZERO) {
        const int forced = g_force_path.load(std::memory_order_relaxed);
        if (forced != 0) {
            if (!path_serves(forced, path, p.in_dtype, p.M)) return TG_ERR_UNSUPPORTED;
            path = forced;
        }
    }

    DeviceState* ds = nullptr;
    tg_status st = device_state(&ds);
    if (st != TG_OK) return st;

    tg::GemmArgs a;
    a.M = static_cast<int>(p.M);
    a.N = static_cast<int>(p.N);
    a.K = static_cast<int>(p.K);
    a.batch = static_cast<int>(p.batch);
    a.sA = p.batch > 1 ? p.sA : 0;
    a.sB = p.batch > 1 ? p.sB : 0;
    a.sC = p.batch > 1 ? p.sC : 0;
    a.A = p.A;
    a.lda = p.lda;
    a.B = p.B;
    a.ldb = p.ldb;
    a.C = p.C;
    a.ldc = p.ldc;
    a.out_f32 = (p.out_dtype == TG_F32);
    a.in_es = p.in_dtype == TG_E4M3 ? 1 : 2;
    a.err = ds->err;
    a.hook = g_test_hook.load(std::memory_order_relaxed);
    a.group_m = g_force_group.load(std::memory_order_relaxed);
    a.split_tail = g_force_split_tail.load(std::memory_order_relaxed);
    a.stages = g_force_stages.load(std::memory_order_relaxed);
    a.num_sms = ds->num_sms;
    a.stream = s;
    a.epi = epi;

    cudaError_t e = cudaSuccess;
    switch (path) {
        case tg::PATH_ZERO: e = tg::launch_epilogue_only(a); break;
        case tg::PATH_SIMT: e = tg::launch_simt_f32(a); break;
        case tg::PATH_MAIN: {
            const int forced_bn = g_force_bn.load(std::memory_order_relaxed);
            int bn = 0, split = 1;
            e = tg::main_plan(a, forced_bn, g_force_split_k.load(std::memory_order_relaxed), &bn,
                              &split);
            if (e != cudaSuccess) break;
            if (a.stages != 0 && a.stages > tg::main_max_stages(bn)) return TG_ERR_UNSUPPORTED;
            a.split_k = split;
            e = tg::launch_main(a, bn);
            break;
        }
        case tg::PATH_BOUNDARY: e = tg::launch_boundary(a); break;
        case tg::PATH_MAIN_PAIR:
            if (a.stages != 0 && a.stages > tg::pair_max_stages()) return TG_ERR_UNSUPPORTED;
            e = tg::launch_main_pair(a);
            break;
        case tg::PATH_SKINNY: e = tg::launch_skinny(a); break;
        default: return TG_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace

namespace tg {

namespace {

// Encoded tensor maps, keyed by every argument of encode_tmap (the encoded
// bytes depend on nothing else: the swizzle, L2 promotion and fill mode are
// fixed).  A call that repeats a previous call's operands (the usual case:
// the same buffers every step) copies 128 bytes instead of encoding again.
// Direct-mapped; a colliding key replaces the entry.  Guarded by a mutex.
struct TmapKey {
    const void* ptr;
    uint64_t cols, rows, ld, batch, stride;
    uint32_t box_cols, box_rows;
    int es;
    int kind;  // 0: operand load map (128-byte swizzle), 1: output store map (no swizzle)
    uint32_t box_chunks;  // > 0: a 4-D operand map of column blocks (kind 0)
    bool operator==(const TmapKey& o) const
    {
        return ptr == o.ptr && cols == o.cols && rows == o.rows && ld == o.ld &&
               batch == o.batch && stride == o.stride && box_cols == o.box_cols &&
               box_rows == o.box_rows && es == o.es && kind == o.kind &&
               box_chunks == o.box_chunks;
    }
};

struct TmapEntry {
    bool used = false;
    TmapKey key{};
    CUtensorMap map{};
};

constexpr int kTmapCacheSize = 1024;
std::mutex g_tmap_mu;
TmapEntry g_tmap_cache[kTmapCacheSize];

uint64_t mix(uint64_t h, uint64_t v)
{
    // splitmix64 finaliser over the running hash
    h ^= v + 0x9e3779b97f4a7c15ULL + (h << 6) + (h >> 2);
    h ^= h >> 30;
    h *= 0xbf58476d1ce4e5b9ULL;
    h ^= h >> 27;
    h *= 0x94d049bb133111ebULL;
    h ^= h >> 31;
    return h;
}

int tmap_slot(const TmapKey& k)
{
    uint64_t h = reinterpret_cast<uintptr_t>(k.ptr);
    h = mix(h, k.cols);
    h = mix(h, k.rows);
    h = mix(h, k.ld);
    h = mix(h, k.batch);
    h = mix(h, k.stride);
    h = mix(h, (static_cast<uint64_t>(k.box_cols) << 32) | k.box_rows);
    h = mix(h, static_cast<uint64_t>(k.es) | (static_cast<uint64_t>(k.kind) << 8) |
                   (static_cast<uint64_t>(k.box_chunks) << 16));
    return static_cast<int>(h % kTmapCacheSize);
}

// Encodes (or finds in the cache) a 3-D map, or with box_chunks > 0 the
// 4-D view described below; kind 0: an operand load map
// (fp16 or byte elements, 128-byte swizzle, 256-byte L2 promotion), kind 1:
// an output store map (fp16 or fp32 elements, no swizzle).
bool encode_map(CUtensorMap* map, int kind, const void* ptr, int es, uint64_t cols, uint64_t rows,
                uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols, uint32_t box_rows,
                uint32_t box_chunks = 0)
{
    if (!g_encode) return false;
    if (kind == 0 ? (es != 1 && es != 2) : (es != 2 && es != 4)) return false;
    if (stride == 0) {
        // one matrix: the third extent is 1 and its stride only has to be a
        // legal value (a multiple of 16 bytes covering the matrix)
        batch = 1;
        stride = (rows * ld * es + 15) / 16 * 16 / es;
    }
    const TmapKey key{ptr, cols, rows, ld, batch, stride, box_cols, box_rows, es, kind, box_chunks};
    const int slot = tmap_slot(key);
    {
        std::lock_guard<std::mutex> lock(g_tmap_mu);
        const TmapEntry& e = g_tmap_cache[slot];
        if (e.used && e.key == key) {
            *map = e.map;
            return true;
        }
    }
    // 3-D: {cols, rows, batch}.  4-D (box_chunks > 0): the same bytes seen
    // as {box_cols, rows, cols / box_cols column blocks, batch}, the block
    // stride box_cols elements, so that one box brings box_chunks adjacent
    // column blocks, each landing as its own [box_rows][box_cols] block
    const uint32_t rank = box_chunks > 0 ? 4 : 3;
    cuuint64_t dims[4] = {cols, rows, batch, 1};
    cuuint64_t strides[3] = {ld * es, stride * es, 0};
    cuuint32_t box[4] = {box_cols, box_rows, 1, 1};
    if (box_chunks > 0) {
        if (cols % box_cols != 0) return false;
        dims[0] = box_cols;
        dims[2] = cols / box_cols;
        dims[3] = batch;
        strides[1] = static_cast<cuuint64_t>(box_cols) * es;
        strides[2] = stride * es;
        box[2] = box_chunks;
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = es == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : es == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = g_encode(map, dt, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          kind == 0 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          kind == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                    : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    TmapEntry& e = g_tmap_cache[slot];
    e.used = true;
    e.key = key;
    e.map = *map;
    return true;
}

}  // namespace

bool encode_tmap(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                 uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                 uint32_t box_rows)
{
    return encode_map(map, 0, ptr, es, cols, rows, ld, batch, stride, box_cols, box_rows);
}

bool encode_tmap_chunks(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                        uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                        uint32_t box_rows, uint32_t box_chunks)
{
    return encode_map(map, 0, ptr, es, cols, rows, ld, batch, stride, box_cols, box_rows,
                      box_chunks);
}

bool encode_tmap_store(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                       uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                       uint32_t box_rows)
{
    return encode_map(map, 1, ptr, es, cols, rows, ld, batch, stride, box_cols, box_rows);
}

// Defined beside the boundary kernel: clusters of S CTAs that share one boundary-kernel
// output tile over K: the largest S of 2, 4, 8 with tiles * S <= num_sms,
// S <= nkb and (given max_clusters[i], the clusters of 2 << i that fit at
// once) `tiles` clusters resident together; else 1.
int boundary_split(long long tiles, int nkb, int num_sms, const int* max_clusters);
}  // namespace tg

extern "C" {

tg_status tg_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                  int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype,
                  tg_stream_t stream)
{
    const Problem p{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, in_dtype, out_dtype};
    int path = tg::PATH_NONE;
    tg_status st = classify(p, &path);
    if (st != TG_OK || path == tg::PATH_NONE) return st;
    return run(path, p, tg::Epilogue{}, stream);
}

tg_status tg_gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A,
                          int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                          int64_t strideB, void* C, int64_t ldc, int64_t strideC,
                          tg_dtype in_dtype, tg_dtype out_dtype, tg_stream_t stream)
{
    const Problem p{batch, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                    in_dtype, out_dtype};
    int path = tg::PATH_NONE;
    tg_status st = classify(p, &path);
    if (st != TG_OK || path == tg::PATH_NONE) return st;
    return run(path, p, tg::Epilogue{}, stream);
}

tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, void* C, int64_t ldc, tg_dtype in_dtype, tg_dtype out_dtype,
                     float alpha, float beta, const void* D, int64_t ldd, const float* bias,
                     tg_activation act, tg_stream_t stream)
{
    if (act != TG_ACT_NONE && act != TG_ACT_RELU && act != TG_ACT_GELU) return TG_ERR_INVALID_ARG;
    const Problem p{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, in_dtype, out_dtype};
    int path = tg::PATH_NONE;
    tg_status st = classify(p, &path);
    if (st != TG_OK || path == tg::PATH_NONE) return st;
    tg::Epilogue epi;
    st = classify_epilogue(M, N, C, ldc, out_dtype, alpha, beta, D, ldd, bias,
                           static_cast<int>(act), &epi);
    if (st != TG_OK) return st;
    return run(path, p, epi, stream);
}

}  // extern "C"

namespace {

// tg_attention_ws with the kernel override passed in (read once by the
// caller, so that every decision of one call sees the same value).
tg_status attention_impl(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                         const void* Q, int64_t ldq, int64_t strideQ, const void* K, int64_t ldk,
                         int64_t strideK, const void* V, int64_t ldv, int64_t strideV, void* O,
                         int64_t ldo, int64_t strideO, float scale, tg_dtype in_dtype,
                         tg_dtype out_dtype, void* workspace, size_t workspace_bytes,
                         tg_stream_t stream, int forced)
{
    if (batch < 0 || Nq < 0 || Nk < 0 || d < 0 || dv < 0) return TG_ERR_INVALID_ARG;
    if (strideQ < 0 || strideK < 0 || strideV < 0 || strideO < 0) return TG_ERR_INVALID_ARG;
    if (in_dtype != TG_F16 || (out_dtype != TG_F16 && out_dtype != TG_F32))
        return TG_ERR_UNSUPPORTED;
    if (Nq > kMaxDim || Nk > kMaxDim || d > kMaxDim || dv > 65535LL * 128 || batch > kMaxBatch)
        return TG_ERR_UNSUPPORTED;
    if (batch == 0 || Nq == 0 || dv == 0) return TG_OK;
    // softmax over no keys, or over all-zero logits of an empty dot product,
    // is not an attention problem
    if (Nk == 0 || d == 0) return TG_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O || ldq < d || ldk < d || ldv < dv || ldo < dv)
        return TG_ERR_INVALID_ARG;
    const size_t eo = esize(out_dtype);
    if (reinterpret_cast<uintptr_t>(O) % eo != 0) return TG_ERR_INVALID_ARG;
    if (batch > 1 && strideO < (Nq - 1) * ldo + dv) return TG_ERR_INVALID_ARG;
    u128 o0, o1, q0, q1, k0, k1, v0, v1;
    span(O, Nq, dv, ldo, eo, &o0, &o1, batch, strideO);
    span(Q, Nq, d, ldq, 2, &q0, &q1, batch, strideQ);
    span(K, Nk, d, ldk, 2, &k0, &k1, batch, strideK);
    span(V, Nk, dv, ldv, 2, &v0, &v1, batch, strideV);
    const u128 top = static_cast<u128>(1) << 64;
    if (o1 > top || q1 > top || k1 > top || v1 > top) return TG_ERR_INVALID_ARG;
    if (overlaps(o0, o1, q0, q1) || overlaps(o0, o1, k0, k1) || overlaps(o0, o1, v0, v1))
        return TG_ERR_INVALID_ARG;
    // Q, K and V are read by the TMA engine only
    auto tma_ok = [&](const void* p, int64_t ld, int64_t stride, int64_t rows) {
        return reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 8 == 0 &&
               ld < (int64_t(1) << 38) && (batch == 1 || tma_stride_ok(stride, rows, ld, 2));
    };
    if (!tma_ok(Q, ldq, strideQ, Nq) || !tma_ok(K, ldk, strideK, Nk) || !tma_ok(V, ldv, strideV, Nk))
        return TG_ERR_UNSUPPORTED;

    if (workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return TG_ERR_INVALID_ARG;

    DeviceState* ds = nullptr;
    tg_status st = device_state(&ds);
    if (st != TG_OK) return st;
    // a split over the keys when the grid is small and the caller's
    // workspace holds its partial results
    const size_t need = tg::attention_ws_bytes(static_cast<int>(batch), static_cast<int>(Nq),
                                               static_cast<int>(Nk), static_cast<int>(dv),
                                               ds->num_sms);
    const bool ws_ok = need > 0 && workspace != nullptr && workspace_bytes >= need;
    const int choice = tg::attention_kernel_choice(
        static_cast<int>(batch), static_cast<int>(Nq), static_cast<int>(Nk), static_cast<int>(d),
        static_cast<int>(dv), ds->num_sms, ws_ok, forced);
    const bool split = choice == 2;
    // the P-in-TMEM kernel cuts the tiles of a short last wave in two along
    // the keys when the workspace holds the halves' partial results
    size_t need_tail = 0;
    if (choice == 3 && workspace != nullptr) {
        need_tail = tg::attention_tail_ws_bytes(static_cast<int>(batch), static_cast<int>(Nq),
                                                static_cast<int>(Nk), ds->num_sms);
        if (workspace_bytes < need_tail) need_tail = 0;
    }
    const size_t used = split ? need : need_tail;
    if (used > 0) {
        u128 w0 = static_cast<u128>(reinterpret_cast<uintptr_t>(workspace));
        u128 w1 = w0 + used;
        if (w1 > top || overlaps(w0, w1, o0, o1) || overlaps(w0, w1, q0, q1) ||
            overlaps(w0, w1, k0, k1) || overlaps(w0, w1, v0, v1))
            return TG_ERR_INVALID_ARG;
    }
    tg::AttnArgs a;
    a.batch = static_cast<int>(batch);
    a.Nq = static_cast<int>(Nq);
    a.Nk = static_cast<int>(Nk);
    a.d = static_cast<int>(d);
    a.dv = static_cast<int>(dv);
    a.Q = Q;
    a.ldq = ldq;
    a.sQ = batch > 1 ? strideQ : 0;
    a.K = K;
    a.ldk = ldk;
    a.sK = batch > 1 ? strideK : 0;
    a.V = V;
    a.ldv = ldv;
    a.sV = batch > 1 ? strideV : 0;
    a.O = O;
    a.ldo = ldo;
    a.sO = batch > 1 ? strideO : 0;
    a.out_f32 = out_dtype == TG_F32;
    a.scale = scale;
    a.err = ds->err;
    a.hook = g_test_hook.load(std::memory_order_relaxed);
    a.stream = static_cast<cudaStream_t>(stream);
    if (split) {
        a.n_split = tg::attention_splits(a.batch, a.Nq, a.Nk, a.dv, ds->num_sms);
        a.ws = workspace;
    }
    a.tmem_p = choice == 3;
    if (need_tail > 0) {
        a.tail_tiles = tg::attention_tail_plan(a.batch, a.Nq, a.Nk, ds->num_sms, &a.tail_pieces);
        a.ws = workspace;
    }
    return tg::launch_attention(a) == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

bool attention_sizes_ok(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv)
{
    if (batch <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || dv <= 0) return false;
    return !(Nq > kMaxDim || Nk > kMaxDim || d > kMaxDim || dv > 65535LL * 128 ||
             batch > kMaxBatch);
}

// tg_attention_workspace_size with the kernel override passed in.
size_t workspace_size_impl(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                           int forced)
{
    if (!attention_sizes_ok(batch, Nq, Nk, d, dv)) return 0;
    DeviceState* ds = nullptr;
    if (device_state(&ds) != TG_OK) return 0;
    const size_t split = tg::attention_ws_bytes(static_cast<int>(batch), static_cast<int>(Nq),
                                                static_cast<int>(Nk), static_cast<int>(dv),
                                                ds->num_sms);
    const int choice = tg::attention_kernel_choice(
        static_cast<int>(batch), static_cast<int>(Nq), static_cast<int>(Nk), static_cast<int>(d),
        static_cast<int>(dv), ds->num_sms, split > 0, forced);
    if (choice == 2) return split;
    if (choice == 3)
        return tg::attention_tail_ws_bytes(static_cast<int>(batch), static_cast<int>(Nq),
                                           static_cast<int>(Nk), ds->num_sms);
    return 0;
}

// tg_attention_kernel with the kernel override passed in.
int kernel_choice_impl(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                       int split_allowed, int forced)
{
    if (!attention_sizes_ok(batch, Nq, Nk, d, dv)) return 0;
    DeviceState* ds = nullptr;
    if (device_state(&ds) != TG_OK) return 0;
    const bool ws_ok = split_allowed != 0 &&
                       tg::attention_ws_bytes(static_cast<int>(batch), static_cast<int>(Nq),
                                              static_cast<int>(Nk), static_cast<int>(dv),
                                              ds->num_sms) > 0;
    return tg::attention_kernel_choice(static_cast<int>(batch), static_cast<int>(Nq),
                                       static_cast<int>(Nk), static_cast<int>(d),
                                       static_cast<int>(dv), ds->num_sms, ws_ok, forced);
}

}  // namespace

extern "C" {

tg_status tg_attention_ws(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                          const void* Q, int64_t ldq, int64_t strideQ, const void* K, int64_t ldk,
                          int64_t strideK, const void* V, int64_t ldv, int64_t strideV, void* O,
                          int64_t ldo, int64_t strideO, float scale, tg_dtype in_dtype,
                          tg_dtype out_dtype, void* workspace, size_t workspace_bytes,
                          tg_stream_t stream)
{
    return attention_impl(batch, Nq, Nk, d, dv, Q, ldq, strideQ, K, ldk, strideK, V, ldv, strideV,
                          O, ldo, strideO, scale, in_dtype, out_dtype, workspace, workspace_bytes,
                          stream, g_force_attn.load(std::memory_order_relaxed));
}

tg_status tg_attention(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                       const void* Q, int64_t ldq, int64_t strideQ, const void* K, int64_t ldk,
                       int64_t strideK, const void* V, int64_t ldv, int64_t strideV, void* O,
                       int64_t ldo, int64_t strideO, float scale, tg_dtype in_dtype,
                       tg_dtype out_dtype, tg_stream_t stream)
{
    return tg_attention_ws(batch, Nq, Nk, d, dv, Q, ldq, strideQ, K, ldk, strideK, V, ldv,
                           strideV, O, ldo, strideO, scale, in_dtype, out_dtype, nullptr, 0,
                           stream);
}

tg_status tg_attention_noalloc(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                               const void* Q, int64_t ldq, int64_t strideQ, const void* K,
                               int64_t ldk, int64_t strideK, const void* V, int64_t ldv,
                               int64_t strideV, void* O, int64_t ldo, int64_t strideO, float scale,
                               tg_dtype in_dtype, tg_dtype out_dtype, tg_stream_t stream)
{
    // one read of the override: the need, the choice below and the launch
    // all see the same kernel selection
    const int forced = g_force_attn.load(std::memory_order_relaxed);
    const size_t need = workspace_size_impl(batch, Nq, Nk, d, dv, forced);
    if (need == 0)  // no split (or invalid arguments, which attention_impl reports)
        return attention_impl(batch, Nq, Nk, d, dv, Q, ldq, strideQ, K, ldk, strideK, V, ldv,
                              strideV, O, ldo, strideO, scale, in_dtype, out_dtype, nullptr, 0,
                              stream, forced);
    size_t bytes = 0;
    void* scratch = tg::attention_static_scratch(&bytes);
    if (scratch == nullptr) return TG_ERR_CUDA;
    if (need > bytes) {
        // the key split needs more than the static scratch; a split of the
        // last wave only saves time, and the call runs without it
        if (kernel_choice_impl(batch, Nq, Nk, d, dv, 1, forced) != 3) return TG_ERR_UNSUPPORTED;
        return attention_impl(batch, Nq, Nk, d, dv, Q, ldq, strideQ, K, ldk, strideK, V, ldv,
                              strideV, O, ldo, strideO, scale, in_dtype, out_dtype, nullptr, 0,
                              stream, forced);
    }
    return attention_impl(batch, Nq, Nk, d, dv, Q, ldq, strideQ, K, ldk, strideK, V, ldv, strideV,
                          O, ldo, strideO, scale, in_dtype, out_dtype, scratch, bytes, stream,
                          forced);
}

size_t tg_attention_workspace_size(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv)
{
    return workspace_size_impl(batch, Nq, Nk, d, dv, g_force_attn.load(std::memory_order_relaxed));
}

int tg_attention_kernel(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                        int split_allowed)
{
    return kernel_choice_impl(batch, Nq, Nk, d, dv, split_allowed,
                              g_force_attn.load(std::memory_order_relaxed));
}

int tg_attention_tail_plan(int64_t batch, int64_t Nq, int64_t Nk, int64_t d, int64_t dv,
                           int num_sms, int* pieces)
{
    int p = 0;
    int tail = 0;
    if (batch > 0 && Nq > 0 && Nk > 0 && d > 0 && dv > 0 && num_sms > 0 && Nq <= kMaxDim &&
        Nk <= kMaxDim && batch <= kMaxBatch &&
        tg::attention_tmem_p_serves(static_cast<int>(d), static_cast<int>(dv)))
        tail = tg::attention_tail_plan(static_cast<int>(batch), static_cast<int>(Nq),
                                       static_cast<int>(Nk), num_sms, &p);
    if (pieces != nullptr) *pieces = tail > 0 ? p : 0;
    return tail;
}

tg_status tg_attention_force_kernel(int kernel)
{
    if (!(kernel == 0 || kernel == 1 || kernel == 3)) return TG_ERR_INVALID_ARG;
    g_force_attn.store(kernel, std::memory_order_relaxed);
    return TG_OK;
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
    return tg_gemm_batched_path(1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, in_dtype, out_dtype);
}

int tg_gemm_batched_path(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A,
                         int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                         int64_t strideB, void* C, int64_t ldc, int64_t strideC,
                         tg_dtype in_dtype, tg_dtype out_dtype)
{
    const Problem p{batch, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                    in_dtype, out_dtype};
    int path = tg::PATH_NONE;
    if (classify(p, &path) != TG_OK) return tg::PATH_NONE;
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

tg_status tg_gemm_force_stages(int stages)
{
    if (stages != 0 && (stages < 2 || stages > 8)) return TG_ERR_INVALID_ARG;
    g_force_stages.store(stages, std::memory_order_relaxed);
    return TG_OK;
}

tg_status tg_gemm_force_split_k(int split)
{
    if (split != 0 && split != 1 && split != 2 && split != 4 && split != 8)
        return TG_ERR_INVALID_ARG;
    g_force_split_k.store(split, std::memory_order_relaxed);
    return TG_OK;
}

int tg_gemm_main_plan(int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in_dtype,
                      int num_sms, int* bn)
{
    if (M <= 0 || N <= 0 || K <= 0 || batch <= 0 || num_sms <= 0 || M > INT32_MAX ||
        N > INT32_MAX || K > INT32_MAX || batch > INT32_MAX ||
        (in_dtype != TG_F16 && in_dtype != TG_E4M3)) {
        if (bn != nullptr) *bn = 0;
        return 0;
    }
    int w = 0, split = 1;
    tg::main_plan_host(M, N, K, batch, in_dtype == TG_E4M3 ? 1 : 2, num_sms, &w, &split);
    if (bn != nullptr) *bn = w;
    return split;
}

tg_status tg_gemm_force_split_tail(int tiles)
{
    if (tiles < -1) return TG_ERR_INVALID_ARG;
    g_force_split_tail.store(tiles, std::memory_order_relaxed);
    return TG_OK;
}

int tg_gemm_pair_split_tail(int64_t tiles, int max_pairs)
{
    if (tiles <= 0 || max_pairs <= 0 || tiles >= (int64_t(1) << 31)) return 0;
    return tg::pair_split_tail(static_cast<int>(tiles), max_pairs, -1);
}

int tg_gemm_boundary_split(int64_t tiles, int kblocks, int num_sms)
{
    if (tiles <= 0 || kblocks <= 0 || num_sms <= 0) return 1;
    return tg::boundary_split(tiles, kblocks, num_sms, nullptr);
}

int tg_gemm_version(void) { return 100; }

}  // extern "C"

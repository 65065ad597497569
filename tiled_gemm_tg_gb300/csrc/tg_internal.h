// tg_internal.h -- host-side interface between the C-ABI dispatcher and the
// kernel launchers.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tg {

enum Path : int {
    PATH_NONE = 0,
    PATH_ZERO = 1,      // K == 0: C is the empty sum
    PATH_SIMT = 2,      // fp32 register-blocked SIMT kernel
    PATH_MAIN = 3,      // TMA + tcgen05 warp-specialised persistent kernel
    PATH_BOUNDARY = 4,  // tcgen05 kernel with predicated (non-TMA) loads
    PATH_SKINNY = 5,    // small M: swapped operands, split-K over a cluster
    PATH_MAIN_PAIR = 6, // TMA + tcgen05, 256 x 256 tiles on CTA pairs (cta_group::2)
};

// Programmatic dependent launch (on by default): a kernel's prologue (barrier
// setup, TMEM allocation, descriptor prefetch) may overlap the end of the
// kernel before it on the stream; the kernel waits for that grid's
// completion (griddepcontrol.wait) before touching global memory.
#ifndef TG_PDL
#define TG_PDL 1
#endif

inline void set_pdl_attr(cudaLaunchAttribute& at)
{
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = TG_PDL;
}

// Bits of the device error word (OR-ed by kernels that abandon a wait).
enum ErrBits : unsigned int {
    ERR_MAIN_PRODUCER = 1u << 0,
    ERR_MAIN_MMA = 1u << 1,
    ERR_MAIN_EPILOGUE = 1u << 2,
    ERR_BOUNDARY = 1u << 3,
    ERR_SKINNY = 1u << 4,
    ERR_DRAIN = 1u << 5,
    ERR_ATTENTION = 1u << 6,
};

// Fused epilogue  C = act(alpha * acc + beta * D + bias[n]), applied to the
// fp32 accumulator before the output conversion.  `on` is 0 for the plain
// store (alpha 1, beta 0, no bias, no activation); kernels then take exactly
// the code path of the unfused call.
enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2 };

struct Epilogue {
    float alpha = 1.0f;
    float beta = 0.0f;
    const void* D = nullptr;     // M x N, the output's element type; read only if beta != 0
    long long ldd = 0;           // row stride of D in elements
    const float* bias = nullptr; // N values, or null
    int act = ACT_NONE;
    int on = 0;
    int d_vec = 0;     // D's base and row stride allow 16-byte loads
    int bias_vec = 0;  // bias is 16-byte aligned
};

// What a kernel needs to walk a strided batch: the number of matrices,
// whether A and B advance with the batch index (1) or are broadcast (0), and
// the matrix strides in elements (the TMA kernels read sA and sB from their
// tensor maps instead).
struct BatchArgs {
    int count = 1;
    int za = 0;
    int zb = 0;
    long long sA = 0, sB = 0, sC = 0;
};

struct GemmArgs {
    int M, N, K;
    // Strided batch: matrix b of X starts at X + b * sX elements; a stride of
    // 0 broadcasts one matrix to every b.  batch == 1 for a single GEMM.
    int batch = 1;
    long long sA = 0, sB = 0, sC = 0;
    const void* A;
    long long lda;
    const void* B;
    long long ldb;
    void* C;
    long long ldc;
    bool out_f32;
    int in_es = 2;      // input element size: 2 (fp16) or 1 (E4M3)
    unsigned int* err;  // device error word
    int hook;           // test hook (0 = off), see tg_gemm_test_hook
    int group_m;        // grouped tile-order height, 0 = the kernel's default
    int split_tail = -1;  // pair kernel: tiles of the last wave cut in two, -1 = automatic
    int stages = 0;       // TMA kernels: pipeline stages in the ring, 0 = the kernel's most
    int split_k = 1;      // one-CTA kernel: CTAs sharing each tile over K (a cluster)
    int num_sms;
    cudaStream_t stream;
    Epilogue epi;

    BatchArgs batch_args() const
    {
        BatchArgs b;
        b.count = batch;
        b.za = sA != 0 ? 1 : 0;
        b.zb = sB != 0 ? 1 : 0;
        b.sA = sA;
        b.sB = sB;
        b.sC = sC;
        return b;
    }
};

// Encodes a 3-D tensor map over `batch` row-major matrices of `es`-byte
// elements (2: fp16, 1: E4M3 bytes; inner extent `cols`, `rows` rows, row
// stride `ld` elements, matrix stride `stride` elements; stride 0 maps a
// single matrix that every batch coordinate must address as z = 0) with a box
// of box_cols x box_rows x 1 and 128-byte swizzle.  Returns false if the
// driver rejects it.
bool encode_tmap(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                 uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                 uint32_t box_rows);

// The same bytes as a 4-D map {box_cols, rows, cols / box_cols, batch} whose
// box {box_cols, box_rows, box_chunks, 1} brings box_chunks adjacent
// column blocks in one copy, block j landing box_rows * box_cols elements
// after block j - 1.  cols must be a multiple of box_cols (no block may end
// past the last column: such a box would read beyond the matrix).
bool encode_tmap_chunks(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                        uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                        uint32_t box_rows, uint32_t box_chunks);

// The same for an output written by TMA stores: es = 2 (fp16) or 4 (fp32),
// no swizzle, box_cols x box_rows x 1.
bool encode_tmap_store(CUtensorMap* map, const void* ptr, int es, uint64_t cols, uint64_t rows,
                       uint64_t ld, uint64_t batch, uint64_t stride, uint32_t box_cols,
                       uint32_t box_rows);

cudaError_t launch_simt_f32(const GemmArgs& a);
cudaError_t launch_main(const GemmArgs& a, int bn);
cudaError_t launch_main_pair(const GemmArgs& a);
cudaError_t launch_boundary(const GemmArgs& a);
cudaError_t launch_skinny(const GemmArgs& a);
// K == 0: C = act(beta * D + bias) elementwise (zeros without an epilogue),
// for every matrix of a strided batch.
cudaError_t launch_epilogue_only(const GemmArgs& a);

// Attention forward O_b = softmax(scale * Q_b K_b^T) V_b for a strided batch
// (fp16 Q, K, V; fp16 or fp32 O).  Strides and row strides in elements.
struct AttnArgs {
    int batch, Nq, Nk, d, dv;
    const void* Q;
    long long ldq, sQ;
    const void* K;
    long long ldk, sK;
    const void* V;
    long long ldv, sV;
    void* O;
    long long ldo, sO;
    bool out_f32;
    float scale;
    unsigned int* err;
    int hook;
    cudaStream_t stream;
    // a split over the keys (n_split > 1) writes partial results to `ws`
    // (attention_ws_bytes of them) and merges them in a second kernel
    int n_split = 1;
    void* ws = nullptr;
    // the kernel that keeps P in tensor memory (attention_fwd2.cu); needs
    // d <= 128, dv <= 128 and no key split
    bool tmem_p = false;
    // with tmem_p: the tiles of the last wave each cut into `tail_pieces`
    // ranges of the keys and merged in the kernel, through `ws`
    // (attention_tail_plan, attention_tail_ws_bytes)
    int tail_tiles = 0;
    int tail_pieces = 0;
};

cudaError_t launch_attention(const AttnArgs& a);
// How many key splits the attention forward uses on `num_sms` SMs (1: none),
// the workspace bytes they need, and the offset (in floats) of the
// maxima/normalisers after the O partials.
int attention_splits(int batch, int Nq, int Nk, int dv, int num_sms);
size_t attention_ws_bytes(int batch, int Nq, int Nk, int dv, int num_sms);
long long attention_ws_o_floats(int batch, int Nq, int dv, int n_split);
// The current device's address of the file-scope attention scratch (looked
// up once per device) and its size; nullptr on failure.
void* attention_static_scratch(size_t* bytes);
// The forward kernel that keeps P in tensor memory: whether it serves these
// head sizes, and its launch.
bool attention_tmem_p_serves(int d, int dv);
cudaError_t launch_attention_tmem_p(const AttnArgs& a);
// Its tail split: how many tiles of a last, partial wave are cut in two
// (0: none), the workspace that needs, and the workspace's layout (O rows,
// then maxima and normalisers, then one counter per tail tile).
int attention_tail_plan(int batch, int Nq, int Nk, int num_sms, int* pieces);
size_t attention_tail_ws_bytes(int batch, int Nq, int Nk, int num_sms);
long long attention_tail_o_floats(int tail, int pieces);
long long attention_tail_ml_floats(int tail, int pieces);
// Which forward kernel a call runs: 1 the general kernel (any d, dv), 2 the
// same with the keys split over CTAs (only when `split_ok`: the caller's
// workspace holds the partials), 3 the kernel that keeps P in tensor memory
// (d <= 128, dv <= 128).  `forced` is 0 (automatic), 1 or 3.
int attention_kernel_choice(int batch, int Nq, int Nk, int d, int dv, int num_sms, bool split_ok,
                            int forced);

// Tile width the main kernel uses for this problem (64, 128 or 256).
int main_tile_n(int M, int N, int batch, int num_sms);
// Tile width and split over K of the main kernel for the call `a`: a
// forced tile width (0: automatic) and split (0: automatic), else the
// default width unsplit or, when the tiles leave half the SMs idle, a wider
// or equal tile split over a cluster if that is estimated faster (every
// cluster resident at once).  main_plan_host: the same without the
// residency check, on the host alone.
cudaError_t main_plan(const GemmArgs& a, int forced_bn, int forced_split, int* bn, int* split);
void main_plan_host(long long M, long long N, long long K, long long batch, int es, int num_sms,
                    int* bn, int* split);
// The most pipeline stages (the default ring) of the one-CTA kernel with
// tile width bn, and of the pair kernel.
int main_max_stages(int bn);
int pair_max_stages();

// Largest M the skinny kernel serves.
constexpr int kSkinnyMaxM = 64;

// Number of 256 x 256 tiles the pair kernel would compute.
int pair_tiles(int M, int N);
// How many of the pair kernel's `total` tiles (the last ones) it cuts into
// two 256 x 128 halves on `max_pairs` co-resident CTA pairs: the whole last
// wave when twice its tiles fit in one wave, else none; `forced` >= 0
// overrides the choice (capped at total).
int pair_split_tail(int total, int max_pairs, int forced);

// The pair kernel takes over once a problem (all products of a batch
// together) has enough 256 x 256 tiles for its longer pipeline fill to pay:
// at least kPairMinTiles with K >= kPairLongK, or kPairMinTilesShortK with
// K >= kPairMinK, and M, N >= 512.  Measured with the configuration sweep
// (CUDA-graph replay): the one-CTA kernel with 128 x 256 tiles wins at 64
// and 128 pair tiles with K <= 2048 (2048 x 2048 x 1024: 10.9 against 12.8
// us; 2048^3: 16.7 against 17.5; 4096 x 2048 x 1024: 17.6 against 18.1), the
// pair kernel at 64 tiles with K = 4096 (2048 x 2048 x 4096: 26.4 against
// 28.1) and from 144 tiles (3072 x 3072 x 2048: 28.0 against 29.7; 4096 x
// 4096 x 1024: 27.1 against 31.2); below K = 1024 the one-CTA kernel's
// shorter fill wins everywhere (8192 x 8192 x 512: 71.5 against 80.3 us).
constexpr int kPairMinTiles = 64;
constexpr int kPairMinTilesShortK = 144;
constexpr int kPairLongK = 4096;
constexpr int kPairMinK = 1024;
constexpr int kPairMinMN = 512;

}  // namespace tg
